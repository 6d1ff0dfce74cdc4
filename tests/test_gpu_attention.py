"""GPU parity of the causal attention core (tcgen05 kernels) against the float64 oracle.

Per-step ops on seeded bf16 inputs: the forward (a and the row statistics it
keeps) and the backward (dq, dk, dv).  Shapes cover one and several 128-row
blocks, ragged token counts, sequences shorter than the microbatch, grouped
K/V heads (groups of 1, 2, 3, 4 and 8 query heads: odd groups run the
one-tile forward, even ones the two-tile forward) and both head sizes.  The backward reads the GPU forward's a and
row statistics, as the stage does.  Bar per step: relative Frobenius <= 5e-3,
max-abs <= 2e-2 max|ref| (tests/parity.py).
"""
import numpy as np
import pytest
import torch

from backward_split_linear_gb300 import binding as zb
from backward_split_linear_gb300 import synth
from backward_split_linear_gb300.runtime import Stage, bf16_from_bits, f64_from_bf16
from oracle import stage as S
from parity import CAUSAL_MAX_TOL, assert_close, causal_stage_fro_tol, draw_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _status_clean(cuda_device):
    zb.zb_device_status(reset=True)
    yield
    st, code = zb.zb_device_status()
    assert st == 0, f"device status word set: {code}"


def run_forward(qkvb, t, nh, nkv, d, seq_len):
    qkv = bf16_from_bits(qkvb)
    a = torch.full((t, nh * d), float("nan"), dtype=torch.bfloat16, device="cuda")
    stride = zb.zb_op_attention_stat_stride(t)
    lse = torch.zeros(nh, stride, dtype=torch.float32, device="cuda")
    zb.zb_op_attention_causal_forward(qkv, a, lse, t, nh, nkv, d, seq_len)
    return qkv, a, lse


def run_backward(qkv, a, lse, dab, t, nh, nkv, d, seq_len):
    da = bf16_from_bits(dab)
    dvec = torch.zeros_like(lse)
    dqkv = torch.full((t, (nh + 2 * nkv) * d), float("nan"), dtype=torch.bfloat16, device="cuda")
    zb.zb_op_attention_causal_backward(qkv, a, da, lse, dvec, dqkv, t, nh, nkv, d, seq_len)
    return dqkv


SHAPES = [(300, 4, 2, 64, 0), (512, 4, 1, 128, 256), (77, 2, 1, 128, 0), (640, 8, 2, 64, 128),
          (1, 2, 2, 64, 0), (384, 2, 2, 128, 128), (384, 16, 2, 128, 0), (200, 6, 2, 64, 0),
          # the last sequence shorter than seq_len and the token count off the 128-row grid
          (700, 8, 2, 128, 256), (450, 6, 3, 64, 128)]


@pytest.mark.parametrize("t,nh,nkv,d,seq_len", SHAPES)
def test_forward_and_backward(t, nh, nkv, d, seq_len):
    rng = np.random.default_rng(100 + t + d)
    qkvb, qkv64 = draw_bf16(rng, (t, (nh + 2 * nkv) * d))
    dab, da64 = draw_bf16(rng, (t, nh * d))
    qkv, a, lse = run_forward(qkvb, t, nh, nkv, d, seq_len)
    ref_a = S.attention_causal(qkv64, nh, nkv, d, seq_len)
    assert_close(f64_from_bf16(a), ref_a, "attention output a")
    # the row statistic: log2 of sum_k exp(score) over the visible keys, scores scaled by 1/sqrt(d)
    q, k, _ = S._heads(qkv64, nh, nkv, d)
    lse_ref = np.zeros((nh, t))
    for s0, s1 in S.sequences(t, seq_len):
        for h in range(nh):
            sc = (q[s0:s1, h] @ k[s0:s1, h // (nh // nkv)].T) / np.sqrt(d)
            sc = np.where(np.tril(np.ones((s1 - s0, s1 - s0), dtype=bool)), sc, -np.inf)
            mx = sc.max(axis=1)
            lse_ref[h, s0:s1] = (mx + np.log(np.exp(sc - mx[:, None]).sum(axis=1))) / np.log(2.0)
    got_lse = lse.cpu().numpy()[:, :t]
    assert np.max(np.abs(got_lse - lse_ref)) < 2e-2, "row log-sum-exp"
    dqkv = run_backward(qkv, a, lse, dab, t, nh, nkv, d, seq_len)
    ref = S.attention_causal_grad(da64, qkv64, nh, nkv, d, seq_len)
    got = f64_from_bf16(dqkv)
    w = nh * d
    kw = nkv * d
    assert_close(got[:, :w], ref[:, :w], "dq")
    assert_close(got[:, w:w + kw], ref[:, w:w + kw], "dk")
    assert_close(got[:, w + kw:], ref[:, w + kw:], "dv")


@pytest.mark.parametrize("nh", [1, 2])
@pytest.mark.parametrize("d", [64, 128])
def test_rescale_when_row_maxima_rise(d, nh):
    """Scores that grow with the key index make a row's maximum rise by far more than the
    forward's rescale threshold from one key block to the next, for every other query row
    (the rows in between see falling scores): the rescale runs in some rows of a warp and
    not in others.  Checked: a and the row statistic (what the rescale touches) and dv.
    dq and dk are left out on this input: its softmax rows are nearly one-hot, so dS =
    P (dP - D) cancels almost exactly, and D = rowsum(dO * O) from the bf16 output alone
    moves dq by about 5e-2 relative (a float64 replay of that rounding gives the same).
    One head runs the one-tile forward, two heads of one kv head the two-tile forward."""
    t, nkv = 1024, 1
    rng = np.random.default_rng(31 + d)
    u = np.ones(d)
    sign = np.where(np.arange(t) % 2 == 0, 1.0, -1.0)
    q = sign[:, None] * u[None, :] + 0.05 * rng.standard_normal((t, d))
    k = (5.0 * np.arange(t) / t)[:, None] * u[None, :] + 0.05 * rng.standard_normal((t, d))
    v = rng.standard_normal((t, d))
    qkv64 = np.concatenate([q] * nh + [k, v], axis=1)
    qkvb = synth.bf16_bits(qkv64.astype(np.float32))
    qkv64 = synth.bf16_to_f64(qkvb)
    dab, da64 = draw_bf16(rng, (t, nh * d))
    qkv, a, lse = run_forward(qkvb, t, nh, nkv, d, 0)
    assert_close(f64_from_bf16(a), S.attention_causal(qkv64, nh, nkv, d, 0), "a with rising maxima")
    qh, kh, _ = S._heads(qkv64, nh, nkv, d)
    for h in range(nh):
        sc = (qh[:, h] @ kh[:, 0].T) / np.sqrt(d)
        sc = np.where(np.tril(np.ones((t, t), dtype=bool)), sc, -np.inf)
        mx = sc.max(axis=1)
        ref_lse = (mx + np.log(np.exp(sc - mx[:, None]).sum(axis=1))) / np.log(2.0)
        assert np.max(np.abs(lse.cpu().numpy()[h, :t] - ref_lse)) < 2e-2 * max(1.0, np.max(np.abs(ref_lse)))
    dqkv = run_backward(qkv, a, lse, dab, t, nh, nkv, d, 0)
    ref = S.attention_causal_grad(da64, qkv64, nh, nkv, d, 0)
    got = f64_from_bf16(dqkv)
    assert_close(got[:, (nh + nkv) * d :], ref[:, (nh + nkv) * d :], "dv with rising maxima")
    assert np.all(np.isfinite(got))


def test_backward_bitwise_reproducible():
    t, nh, nkv, d = 700, 4, 2, 128
    rng = np.random.default_rng(7)
    qkvb, _ = draw_bf16(rng, (t, (nh + 2 * nkv) * d))
    dab, _ = draw_bf16(rng, (t, nh * d))
    qkv, a, lse = run_forward(qkvb, t, nh, nkv, d, 0)
    outs = [run_backward(qkv, a, lse, dab, t, nh, nkv, d, 0) for _ in range(3)]
    _, a2, lse2 = run_forward(qkvb, t, nh, nkv, d, 0)
    assert torch.equal(a, a2) and torch.equal(lse, lse2)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_full_size_bitwise_reproducible():
    """The 8B-shaped layer (4096 tokens, 32 heads on 8 kv heads, d = 128) run again and again:
    every launch gives the same bits.  The kernels reuse tensor-memory columns that an
    earlier product reads without waiting for it to complete; an MMA that ran out of issue
    order would change results from one launch to the next."""
    t, nh, nkv, d = 4096, 32, 8, 128
    rng = np.random.default_rng(21)
    qkvb, _ = draw_bf16(rng, (t, (nh + 2 * nkv) * d))
    dab, _ = draw_bf16(rng, (t, nh * d))
    qkv, a, lse = run_forward(qkvb, t, nh, nkv, d, 0)
    for _ in range(4):
        _, a2, lse2 = run_forward(qkvb, t, nh, nkv, d, 0)
        assert torch.equal(a.view(torch.int16), a2.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))
    first = run_backward(qkv, a, lse, dab, t, nh, nkv, d, 0).view(torch.int16)
    for _ in range(9):
        assert torch.equal(first, run_backward(qkv, a, lse, dab, t, nh, nkv, d, 0).view(torch.int16))
    assert torch.isfinite(a.float()).all() and torch.isfinite(first.view(torch.bfloat16).float()).all()


def test_full_size_one_group():
    """The 8B-shaped layer's attention at 4096 tokens (32 heads on 8 kv heads, d = 128), in
    the launch configuration the stage uses.  Groups are independent, so the oracle follows
    group 0 (query heads 0-3 and kv head 0) exactly."""
    t, nh, nkv, d = 4096, 32, 8, 128
    rng = np.random.default_rng(11)
    qkvb, qkv64 = draw_bf16(rng, (t, (nh + 2 * nkv) * d))
    dab, da64 = draw_bf16(rng, (t, nh * d))
    qkv, a, lse = run_forward(qkvb, t, nh, nkv, d, 0)
    dqkv = run_backward(qkv, a, lse, dab, t, nh, nkv, d, 0)
    g = nh // nkv
    cols_q = slice(0, g * d)
    cols_k = slice(nh * d, nh * d + d)
    cols_v = slice((nh + nkv) * d, (nh + nkv) * d + d)
    sub = np.concatenate([qkv64[:, cols_q], qkv64[:, cols_k], qkv64[:, cols_v]], axis=1)
    ref_a = S.attention_causal(sub, g, 1, d, 0)
    assert_close(f64_from_bf16(a)[:, : g * d], ref_a, "a, heads 0-3")
    ref = S.attention_causal_grad(da64[:, : g * d], sub, g, 1, d, 0)
    got = f64_from_bf16(dqkv)
    assert_close(got[:, cols_q], ref[:, : g * d], "dq, heads 0-3")
    assert_close(got[:, cols_k], ref[:, g * d : g * d + d], "dk, kv head 0")
    assert_close(got[:, cols_v], ref[:, g * d + d :], "dv, kv head 0")
    assert torch.isfinite(dqkv.float()).all()


def test_dq_tiles_outnumber_the_sms():
    """More (head, query block) tiles than SMs, of mixed lengths (sequences of 1024 tokens: 1 to
    8 key blocks per tile), so that each CTA of the persistent dQ kernel takes several tiles from
    its counter, in an order that depends on timing.  Every column of dqkv against the oracle,
    and three runs bit for bit."""
    t, nh, nkv, d, seq_len = 4096, 8, 2, 128, 1024
    rng = np.random.default_rng(13)
    qkvb, qkv64 = draw_bf16(rng, (t, (nh + 2 * nkv) * d))
    dab, da64 = draw_bf16(rng, (t, nh * d))
    qkv, a, lse = run_forward(qkvb, t, nh, nkv, d, seq_len)
    outs = [run_backward(qkv, a, lse, dab, t, nh, nkv, d, seq_len) for _ in range(3)]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    ref = S.attention_causal_grad(da64, qkv64, nh, nkv, d, seq_len)
    got = f64_from_bf16(outs[0])
    assert_close(got[:, : nh * d], ref[:, : nh * d], "dq")
    assert_close(got[:, nh * d : (nh + nkv) * d], ref[:, nh * d : (nh + nkv) * d], "dk")
    assert_close(got[:, (nh + nkv) * d :], ref[:, (nh + nkv) * d :], "dv")


CAUSAL_TF = dict(kind="transformer", n_layers=2, hidden=256, ffn=512, n_heads=4, n_kv_heads=2, head_dim=64)


@pytest.mark.parametrize("seq_len,tokens", [(0, [300, 128]), (128, [384, 200])])
def test_causal_stage_against_oracle(seq_len, tokens):
    """A two-layer stage with the causal attention core: F -> B -> W per microbatch,
    dx and every weight gradient against the oracle at the causal two-layer stage tolerance.
    Both ways of forming D = rowsum(dO * O) run: a microbatch of 256 tokens or more takes the
    CTA-pair GEMM for the output projection's dgrad, whose epilogue forms D (300, 384); a
    smaller one takes the one-CTA GEMM and the row kernel (128, 200)."""
    c = CAUSAL_TF
    inp = synth.stage_inputs(c["kind"], 2, 256, 512, 4, 2, 64, n_mb=len(tokens), seed=21, tokens_per_mb=tokens)
    st = Stage.from_synth(c["kind"], 2, 256, 512, 4, 2, 64, 1e-5, max(tokens), len(tokens), inp["params"],
                          attention="causal", seq_len=seq_len)
    shp = dict(c, eps=1e-5, attention="causal", seq_len=seq_len)
    orc = S.StageOracle(synth.params_f64(inp["params"]), shp)
    dxs = []
    for i, (xb, dyb) in enumerate(zip(inp["x"], inp["dy"])):
        x, dy = bf16_from_bits(xb), bf16_from_bits(dyb)
        y = torch.empty(x.shape[0], 256, dtype=torch.bfloat16, device="cuda")
        dx = torch.empty_like(y)
        st.forward(i, x, y)
        st.backward_input(i, dy, dx)
        st.backward_weight(i)
        dxs.append(dx)
        orc.forward(i, synth.bf16_to_f64(xb))
        ref_dx = orc.backward_input(i, synth.bf16_to_f64(dyb))
        orc.backward_weight(i)
        assert_close(f64_from_bf16(dx), ref_dx, f"dx[{i}]", fro_tol=causal_stage_fro_tol(2), max_tol=CAUSAL_MAX_TOL)
    st.sync()
    for li in range(2):
        for k, ref in orc.grads[li].items():
            assert_close(st.grads[li][k].cpu().numpy(), ref, f"layer {li} d{k}", fro_tol=causal_stage_fro_tol(2),
                         max_tol=CAUSAL_MAX_TOL)
    st.close()


def test_causal_stage_8b_shaped():
    """Two 8B-shaped layers (hidden 4096, ffn 14336, 32 heads on 8 kv heads, d = 128) with the
    causal core: two microbatches of 256 tokens in sequences of 128, F -> B -> W each, against
    the oracle at the causal two-layer stage tolerance (the oracle follows every token)."""
    c = dict(kind="transformer", n_layers=2, hidden=4096, ffn=14336, n_heads=32, n_kv_heads=8, head_dim=128)
    tokens = [256, 256]
    inp = synth.stage_inputs(c["kind"], 2, 4096, 14336, 32, 8, 128, n_mb=2, seed=23, tokens_per_mb=tokens)
    st = Stage.from_synth(c["kind"], 2, 4096, 14336, 32, 8, 128, 1e-5, 256, 2, inp["params"],
                          attention="causal", seq_len=128)
    orc = S.StageOracle(synth.params_f64(inp["params"]), dict(c, eps=1e-5, attention="causal", seq_len=128))
    for i, (xb, dyb) in enumerate(zip(inp["x"], inp["dy"])):
        x, dy = bf16_from_bits(xb), bf16_from_bits(dyb)
        y = torch.empty(256, 4096, dtype=torch.bfloat16, device="cuda")
        dx = torch.empty_like(y)
        st.forward(i, x, y)
        st.backward_input(i, dy, dx)
        orc.forward(i, synth.bf16_to_f64(xb))
        ref_dx = orc.backward_input(i, synth.bf16_to_f64(dyb))
        assert_close(f64_from_bf16(dx), ref_dx, f"dx[{i}]", fro_tol=causal_stage_fro_tol(2), max_tol=CAUSAL_MAX_TOL)
    st.flush()  # both W in one batched call
    st.sync()
    orc.backward_weight(0)
    orc.backward_weight(1)
    for li in range(2):
        for k, ref in orc.grads[li].items():
            assert_close(st.grads[li][k].cpu().numpy(), ref, f"layer {li} d{k}", fro_tol=causal_stage_fro_tol(2),
                         max_tol=CAUSAL_MAX_TOL)
    st.close()


def test_backward_orders_with_the_callers_stream():
    """The backward forks dQ onto a side stream and joins it back: on a caller's stream, work
    queued before the call (a copy that writes the inputs) must land before either kernel reads,
    and work queued after it (a copy of dqkv) must see every column written.  Nothing is
    synchronised in between; the result must equal the same call on synchronised inputs, bit
    for bit."""
    t, nh, nkv, d = 1024, 8, 2, 128
    rng = np.random.default_rng(7)
    qkvb, _ = draw_bf16(rng, (t, (nh + 2 * nkv) * d))
    dab, _ = draw_bf16(rng, (t, nh * d))
    qkv, a, lse = run_forward(qkvb, t, nh, nkv, d, 0)
    torch.cuda.synchronize()
    ref = run_backward(qkv, a, lse, dab, t, nh, nkv, d, 0)
    torch.cuda.synchronize()

    s = torch.cuda.Stream()
    src_qkv, src_da = qkv.clone(), bf16_from_bits(dab)
    qkv2 = torch.zeros_like(qkv)
    da2 = torch.zeros_like(src_da)
    dvec = torch.zeros_like(lse)
    dqkv = torch.full_like(ref, float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        # a slow producer: many small copies in front of the inputs' final copy
        for _ in range(200):
            qkv2.add_(0)
        qkv2.copy_(src_qkv)
        da2.copy_(src_da)
        zb.zb_op_attention_causal_backward(qkv2, a, da2, lse, dvec, dqkv, t, nh, nkv, d, 0, stream=s)
        out = dqkv.clone()
    s.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
