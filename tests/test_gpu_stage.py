"""Whole-stage GPU tests through the C ABI: F -> B -> W per microbatch, flush, orders.

Parity against the float64 oracle (``oracle.stage.StageOracle``) on the seeded
inputs of ``synth.stage_inputs``.  Whole-stage tolerances grow with depth
(tests/parity.py explains why); single-step tolerances are in test_gpu_ops.py.
Full-size cases compare sampled tokens (every op except the weight
contractions acts per token, so the oracle can follow a few tokens exactly)
and check properties that hold at any size.
"""
import numpy as np
import pytest
import torch

from backward_split_linear_gb300 import binding as zb
from backward_split_linear_gb300 import synth
from backward_split_linear_gb300.runtime import Stage, bf16_from_bits, f64_from_bf16
from oracle import schedule as OS
from oracle import stage as S
from parity import MAX_TOL, assert_close, stage_fro_tol

pytestmark = pytest.mark.gpu

TINY = dict(kind="mlp", n_layers=2, hidden=256, ffn=1024, n_heads=0, n_kv_heads=0, head_dim=0)
SMALL_TF = dict(kind="transformer", n_layers=2, hidden=256, ffn=512, n_heads=4, n_kv_heads=2, head_dim=64)
LLAMA8B = dict(kind="transformer", n_layers=4, hidden=4096, ffn=14336, n_heads=32, n_kv_heads=8, head_dim=128)
LLAMA70B = dict(kind="transformer", n_layers=2, hidden=8192, ffn=28672, n_heads=64, n_kv_heads=8, head_dim=128)
EPS = 1e-5


@pytest.fixture(autouse=True)
def _status_clean(cuda_device):
    zb.zb_device_status(reset=True)
    yield
    st, code = zb.zb_device_status()
    assert st == 0, f"device status word set: {code}"


def shp_of(c):
    return dict(c, eps=EPS)


def make_gpu_stage(c, inp, max_tokens, max_inflight):
    return Stage.from_synth(c["kind"], c["n_layers"], c["hidden"], c["ffn"], c["n_heads"], c["n_kv_heads"],
                            c["head_dim"], EPS, max_tokens, max_inflight, inp["params"])


def run_gpu(st, inp, order):
    """Runs (kind, mb) ops; returns dx per microbatch (device tensors)."""
    xs = [bf16_from_bits(b) for b in inp["x"]]
    dys = [bf16_from_bits(b) for b in inp["dy"]]
    dx = {}
    for kind, mb in order:
        if kind == "F":
            y = torch.empty(xs[mb].shape[0], st.out_dim, dtype=torch.bfloat16, device="cuda")
            st.forward(mb, xs[mb], y)
        elif kind == "B":
            dx[mb] = torch.empty(dys[mb].shape[0], st.hidden, dtype=torch.bfloat16, device="cuda")
            st.backward_input(mb, dys[mb], dx[mb])
        else:
            st.backward_weight(mb)
    st.flush()
    st.sync()
    return dx


def run_oracle(c, inp):
    params = synth.params_f64(inp["params"])
    orc = S.StageOracle(params, shp_of(c))
    dx = []
    for i, (xb, dyb) in enumerate(zip(inp["x"], inp["dy"])):
        orc.forward(i, synth.bf16_to_f64(xb))
        dx.append(orc.backward_input(i, synth.bf16_to_f64(dyb)))
        orc.backward_weight(i)
    return dx, orc.grads


def plain_order(n):
    out = []
    for i in range(n):
        out += [("F", i), ("B", i), ("W", i)]
    return out


def compare_stage(c, st, dx_gpu, dx_ref, grads_ref, fro_tol):
    worst = 0.0
    for i, ref in enumerate(dx_ref):
        fro, _ = assert_close(f64_from_bf16(dx_gpu[i]), ref, f"dx[{i}]", fro_tol=fro_tol, max_tol=MAX_TOL)
        worst = max(worst, fro)
    for li, g in enumerate(grads_ref):
        for k, ref in g.items():
            fro, _ = assert_close(st.grads[li][k].cpu().numpy(), ref, f"layer {li} d{k}", fro_tol=fro_tol,
                                  max_tol=MAX_TOL)
            worst = max(worst, fro)
    return worst


def test_tiny_config():
    """2 SwiGLU-MLP layers, hidden 256, ffn 1024, 128 tokens, m = 4, seed 0."""
    c = TINY
    inp = synth.stage_inputs(c["kind"], 2, 256, 1024, tokens=128, n_mb=4, seed=0)
    st = make_gpu_stage(c, inp, 128, 4)
    order = [(k, i) for k, i in zb.zb_schedule("zbh1", 0, 4, 4)]
    dx = run_gpu(st, inp, order)
    dx_ref, g_ref = run_oracle(c, inp)
    compare_stage(c, st, dx, dx_ref, g_ref, stage_fro_tol(c["n_layers"]))


def test_small_transformer_ragged_tokens():
    c = SMALL_TF
    inp = synth.stage_inputs(c["kind"], 2, 256, 512, 4, 2, 64, n_mb=3, seed=1, tokens_per_mb=[200, 77, 1])
    st = make_gpu_stage(c, inp, 256, 2)
    dx = run_gpu(st, inp, [("F", 0), ("F", 1), ("B", 0), ("B", 1), ("W", 0), ("F", 2), ("B", 2)])
    dx_ref, g_ref = run_oracle(c, inp)
    compare_stage(c, st, dx, dx_ref, g_ref, stage_fro_tol(c["n_layers"]))


def test_llama8b_shaped_stage_short_microbatches():
    """8B-shaped stage (4 layers, 4096 / 14336, 32 / 8 heads) with 128- and 100-token microbatches."""
    c = LLAMA8B
    inp = synth.stage_inputs(c["kind"], 4, 4096, 14336, 32, 8, 128, n_mb=2, seed=0, tokens_per_mb=[128, 100])
    st = make_gpu_stage(c, inp, 128, 2)
    dx = run_gpu(st, inp, plain_order(2))
    dx_ref, g_ref = run_oracle(c, inp)
    compare_stage(c, st, dx, dx_ref, g_ref, stage_fro_tol(c["n_layers"]))


def test_llama70b_shaped_stage_short_microbatch():
    """70B-shaped stage (2 layers, 8192 / 28672, 64 / 8 heads) with one 64-token microbatch."""
    c = LLAMA70B
    inp = synth.stage_inputs(c["kind"], 2, 8192, 28672, 64, 8, 128, n_mb=1, seed=0, tokens=64)
    st = make_gpu_stage(c, inp, 64, 1)
    dx = run_gpu(st, inp, plain_order(1))
    dx_ref, g_ref = run_oracle(c, inp)
    compare_stage(c, st, dx, dx_ref, g_ref, stage_fro_tol(c["n_layers"]))


def sampled_token_check(c, inp, dx_gpu, mb, rows):
    """dx of a few tokens against the oracle run on those tokens alone (exact: per-token ops)."""
    params = synth.params_f64(inp["params"])
    x = synth.bf16_to_f64(inp["x"][mb])[rows]
    dy = synth.bf16_to_f64(inp["dy"][mb])[rows]
    _, saved = S.stage_forward(x, params, shp_of(c))
    ref, _ = S.stage_backward_input(dy, params, saved, shp_of(c))
    got = f64_from_bf16(dx_gpu[mb])[rows]
    assert_close(got, ref, f"sampled dx of microbatch {mb}", fro_tol=stage_fro_tol(c["n_layers"]))


def test_zbh1_stage3_p8_m16_order_full_size():
    """ZB-H1 order of stage 3 (p = 8, m = 16) on the 8B-shaped stage at 4096 tokens:
    runs within the p-microbatch ceiling, gives the same weight gradients bit for bit as
    the 1F1B order, and sampled tokens match the oracle."""
    c = LLAMA8B
    p, m, t = 8, 16, 4096
    inp = synth.stage_inputs(c["kind"], 4, 4096, 14336, 32, 8, 128, tokens=t, n_mb=m, seed=0, gamma="ones")
    st = make_gpu_stage(c, inp, t, p)
    zbh1 = zb.zb_schedule("zbh1", 3, p, m)
    dx = run_gpu(st, inp, zbh1)
    assert st.stats()[1] == OS.peak_in_flight(zbh1) == p
    assert st.stats()[0] == 0
    grads_zb = [{k: v.clone() for k, v in g.items()} for g in st.grads]
    rows = np.array([0, 1, 777, 2048, 4095])
    for mb in (0, 15):
        sampled_token_check(c, inp, dx, mb, rows)
    st.zero_grads()
    one_f1b = zb.zb_schedule("1f1b", 3, p, m)
    dx2 = run_gpu(st, inp, one_f1b)
    assert st.stats()[1] == max(OS.peak_in_flight(one_f1b), p)
    for li in range(4):
        for k in grads_zb[li]:
            assert torch.equal(grads_zb[li][k], st.grads[li][k]), (li, k)
    for mb in range(m):
        assert torch.equal(dx[mb], dx2[mb])
    st.close()


def test_concat_identity_full_size():
    """8B-shaped stage, 4096 tokens: one microbatch vs the same tokens as two microbatches.
    Every op except the weight contractions acts per token, so the two runs compute the same
    dx and dW.  They do not round alike: the 4096-token launches may cut their contraction in
    two (the K split), the 2048-token ones do not, so float32 sums run in another order, a few
    bf16 roundings flip and the flips travel down both layers into the stashed gradients
    that W contracts.  dx and dW are held to the two-layer stage tolerance; the exact
    identity on equal stashes is test_flush_batches_consecutive_full_microbatches."""
    c = dict(LLAMA8B, n_layers=2)
    whole = synth.stage_inputs(c["kind"], 2, 4096, 14336, 32, 8, 128, tokens=4096, n_mb=1, seed=3)
    split = {"params": whole["params"],
             "x": [whole["x"][0][:2048], whole["x"][0][2048:]],
             "dy": [whole["dy"][0][:2048], whole["dy"][0][2048:]]}
    st1 = make_gpu_stage(c, whole, 4096, 1)
    dx1 = run_gpu(st1, whole, plain_order(1))
    st2 = make_gpu_stage(c, split, 2048, 2)
    dx2 = run_gpu(st2, split, [("F", 0), ("F", 1), ("B", 0), ("B", 1), ("W", 1), ("W", 0)])
    assert_close(f64_from_bf16(torch.cat([dx2[0], dx2[1]])), f64_from_bf16(dx1[0]), "dx, two microbatches vs one",
                 fro_tol=stage_fro_tol(2))
    for li in range(2):
        for k in st1.grads[li]:
            a = st1.grads[li][k].double()
            b = st2.grads[li][k].double()
            fro = (torch.linalg.norm(a - b) / torch.linalg.norm(a)).item()
            assert fro < stage_fro_tol(2), (li, k, fro)


@pytest.mark.parametrize("tokens", [512, 1024, 2048, 4096, 8192])
def test_linear_4096x14336_token_sweep(tokens):
    """One linear, in 4096, out 14336, m = 4: dW (float32, accumulated) and dx against the
    oracle on sampled rows; each is a single step, so the single-step tolerance applies."""
    n_in, n_out, m = 4096, 14336, 4
    inp = synth.stage_inputs("linear", 1, n_in, n_out, tokens=tokens, n_mb=m, seed=0)
    st = Stage.from_synth("linear", 1, n_in, n_out, max_tokens=tokens, max_inflight=m,
                          params_bits=inp["params"])
    order = [("F", i) for i in range(m)] + [("B", i) for i in range(m)]
    dx = run_gpu(st, inp, order)  # W runs in the flush, ascending microbatch
    w = synth.bf16_to_f64(inp["params"][0]["w"])
    rng = np.random.default_rng(tokens)
    rows_w = np.sort(rng.choice(n_out, 12, replace=False))
    ref = np.zeros((len(rows_w), n_in))
    for i in range(m):
        x = synth.bf16_to_f64(inp["x"][i])
        dy = synth.bf16_to_f64(inp["dy"][i])
        ref += dy[:, rows_w].T @ x
    assert_close(st.grads[0]["w"][torch.from_numpy(rows_w)].cpu().numpy(), ref, "sampled dW rows")
    rows_x = np.sort(rng.choice(tokens, 12, replace=False))
    for i in (0, m - 1):
        dy = synth.bf16_to_f64(inp["dy"][i])[rows_x]
        assert_close(f64_from_bf16(dx[i])[rows_x], dy @ w, f"sampled dx rows, microbatch {i}")
    st.close()


def test_stage_edge_cases_and_errors():
    c = SMALL_TF
    inp = synth.stage_inputs(c["kind"], 2, 256, 512, 4, 2, 64, n_mb=3, seed=4, tokens_per_mb=[64, 0, 64])
    st = make_gpu_stage(c, inp, 64, 2)
    xs = [bf16_from_bits(b) for b in inp["x"]]
    dys = [bf16_from_bits(b) for b in inp["dy"]]
    y = torch.empty(64, 256, dtype=torch.bfloat16, device="cuda")
    dx = torch.empty(64, 256, dtype=torch.bfloat16, device="cuda")

    def err(fn):
        with pytest.raises(zb.ZBError) as e:
            fn()
        return e.value.name

    st.forward(0, xs[0], y)
    assert err(lambda: st.forward(0, xs[0], y)) == "ZB_ERR_ORDER"          # F twice
    assert err(lambda: st.backward_weight(0)) == "ZB_ERR_ORDER"             # W before B
    assert err(lambda: st.backward_input(5, dys[0], dx)) == "ZB_ERR_NO_MB"
    st.forward(1, xs[1], y)                                                 # empty microbatch
    assert err(lambda: st.forward(2, xs[2], y)) == "ZB_ERR_STASH_FULL"      # 2 slots held
    big = torch.zeros(65, 256, dtype=torch.bfloat16, device="cuda")
    assert err(lambda: zb.zb_stage_forward(st.handle, 7, big, 65, big)) == "ZB_ERR_SHAPE"
    st.backward_input(0, dys[0], dx)
    assert err(lambda: st.backward_input(0, dys[0], dx)) == "ZB_ERR_ORDER"  # B twice
    st.backward_input(1, dys[1], dx)
    assert st.stats()[:2] == (2, 2)
    st.flush()                                                              # W of 0 and 1
    assert st.stats() == (0, 2, 0)
    st.forward(2, xs[2], y)                                                 # slot free again
    st.backward_input(2, dys[2], dx)
    st.flush()
    st.sync()
    ref_dx, g_ref = run_oracle(c, inp)
    for li, g in enumerate(g_ref):
        for k, ref in g.items():
            assert_close(st.grads[li][k].cpu().numpy(), ref, f"d{k}", fro_tol=stage_fro_tol(2))
    st.close()


def test_stage_runs_are_bitwise_reproducible():
    c = TINY
    inp = synth.stage_inputs(c["kind"], 2, 256, 1024, tokens=128, n_mb=4, seed=9)
    st = make_gpu_stage(c, inp, 128, 4)
    run_gpu(st, inp, zb.zb_schedule("1f1b", 1, 4, 4))
    first = [{k: v.clone() for k, v in g.items()} for g in st.grads]
    st.zero_grads()
    run_gpu(st, inp, zb.zb_schedule("zbh1", 1, 4, 4))
    for li in range(2):
        for k in first[li]:
            assert torch.equal(first[li][k], st.grads[li][k])


def test_flush_batches_consecutive_full_microbatches():
    """zb_wgrad_flush runs the pending W of consecutive full stash slots as one W over their
    concatenated tokens (the concatenated-batch identity): it must agree with separate W calls
    to float32 summation order and with the oracle to the stage tolerance.  Microbatch 2 is
    short, so it splits the pending slots into the runs {0, 1}, {2}, {3, 4}."""
    c = SMALL_TF
    tok = [128, 128, 77, 128, 128]
    inp = synth.stage_inputs(c["kind"], 2, 256, 512, 4, 2, 64, n_mb=5, seed=11, tokens_per_mb=tok)
    st_batched = make_gpu_stage(c, inp, 128, 5)
    run_gpu(st_batched, inp, [("F", i) for i in range(5)] + [("B", i) for i in range(5)])  # W in the flush
    st_single = make_gpu_stage(c, inp, 128, 5)
    run_gpu(st_single, inp, [("F", i) for i in range(5)] + [("B", i) for i in range(5)] + [("W", i) for i in range(5)])
    _, g_ref = run_oracle(c, inp)
    for li in range(2):
        for k, ref in g_ref[li].items():
            a = st_batched.grads[li][k].double()
            b = st_single.grads[li][k].double()
            assert (torch.linalg.norm(a - b) / torch.linalg.norm(b)).item() < 1e-5, (li, k)
            assert_close(a.cpu().numpy(), ref, f"flushed d{k}", fro_tol=stage_fro_tol(2))
    assert st_batched.stats()[:1] == (0,)
