"""GPU tests of the K-split GEMM path of the stage runtime.

A stage launches its GEMMs with scratch for a K split of the last wave: when
the 256 x 256 tiles left over after the full waves of CTA pairs would keep at
most half of the pairs busy (and K has at least 96 blocks of 64), each of those
tiles is cut into two K halves computed by different CTA pairs, and the half
that finishes second adds the other's float32 partial.  The per-step ops never
split, so they serve as the unsplit comparison on the same inputs.  The shapes
below split on 76 CTA pairs (256 tiles: 3 full waves and 28 split tiles): B of
a linear with 28672 outputs (K = 28672), W of a 4096 x 4096 weight over 16384
tokens (K = 16384), B of a linear with 6144 outputs (K = 6144, halves of 48
blocks), and a ragged case (4000 tokens, 4032 inputs, 24640 outputs: K = 24640
in 385 blocks, split 192 / 193).  `test_split_rule_applies` checks that on the
host.
"""
import math

import numpy as np
import pytest
import torch

from backward_split_linear_gb300 import binding as zb
from backward_split_linear_gb300 import synth
from backward_split_linear_gb300.runtime import Stage, bf16_from_bits, f64_from_bf16
from oracle import stage as S
from parity import MAX_TOL, assert_close, errors, stage_fro_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _status_clean(cuda_device):
    zb.zb_device_status(reset=True)
    yield
    st, code = zb.zb_device_status()
    assert st == 0, f"device status word set: {code}"


def run_linear_stage(inp, t, n_in, n_out):
    st = Stage.from_synth("linear", 1, n_in, n_out, max_tokens=t, max_inflight=1, params_bits=inp["params"])
    x = bf16_from_bits(inp["x"][0])
    dy = bf16_from_bits(inp["dy"][0])
    y = torch.empty(t, n_out, dtype=torch.bfloat16, device="cuda")
    dx = torch.empty(t, n_in, dtype=torch.bfloat16, device="cuda")
    st.forward(0, x, y)
    st.backward_input(0, dy, dx)
    st.backward_weight(0)
    st.sync()
    dw = st.grads[0]["w"].clone()
    st.close()
    return y, dx, dw


SPLIT_SHAPES = [(4096, 4096, 28672), (16384, 4096, 4096), (4096, 4096, 6144), (4000, 4032, 24640)]


def _splits(m, n, k, pairs=76):
    tiles = math.ceil(m / 256) * math.ceil(n / 256)
    rem = tiles % pairs
    return math.ceil(k / 64) >= 96 and 0 < rem and 2 * rem <= pairs


def test_split_rule_applies():
    """Each shape puts at least one of its stage GEMMs through the split (B is [T, in] over K =
    out; W is [out, in] over K = T), by the launch rule of the GEMM."""
    for t, n_in, n_out in SPLIT_SHAPES:
        assert _splits(t, n_in, n_out) or _splits(n_out, n_in, t), (t, n_in, n_out)


@pytest.mark.parametrize("t,n_in,n_out", SPLIT_SHAPES)
def test_split_matches_unsplit_and_oracle(t, n_in, n_out):
    inp = synth.stage_inputs("linear", 1, n_in, n_out, tokens=t, n_mb=1, seed=11)
    y, dx, dw = run_linear_stage(inp, t, n_in, n_out)
    # the same products through the per-step ops, which never split K
    w = bf16_from_bits(inp["params"][0]["w"])
    x = bf16_from_bits(inp["x"][0])
    dy = bf16_from_bits(inp["dy"][0])
    y_op = torch.empty_like(y)
    dx_op = torch.empty_like(dx)
    dw_op = torch.zeros_like(dw)
    zb.zb_op_linear_forward(x, w, None, y_op, t, n_in, n_out)
    zb.zb_op_backward_input(dy, w, dx_op, t, n_in, n_out)
    zb.zb_op_backward_weight(dy, x, dw_op, t, n_in, n_out)
    torch.cuda.synchronize()
    # bf16 results differ from the unsplit ones only where the float32 sum,
    # taken in another order, rounds to a neighbouring bf16 value
    for name, a, b in (("y", y, y_op), ("dx", dx, dx_op)):
        fro, mx = errors(f64_from_bf16(a), f64_from_bf16(b))
        print(f"{name} split vs unsplit: frobenius {fro:.2e}, max {mx:.2e}")
        assert fro < 1e-3 and mx < 1e-2, name
    fro, _ = errors(dw.cpu().numpy(), dw_op.cpu().numpy())
    print(f"dw split vs unsplit: frobenius {fro:.2e}")
    # float32 sums of K = t terms taken in another order: about sqrt(K) 2^-24 apart
    assert fro < 3 * math.sqrt(t) * 2.0 ** -24
    # against the float64 oracle on sampled rows (each row is an exact small product)
    wf = synth.bf16_to_f64(inp["params"][0]["w"])
    xf = synth.bf16_to_f64(inp["x"][0])
    dyf = synth.bf16_to_f64(inp["dy"][0])
    rng = np.random.default_rng(t + n_out)
    rows = np.sort(np.append(rng.choice(t, 15, replace=False), t - 1))
    assert_close(f64_from_bf16(y)[rows], xf[rows] @ wf.T, "sampled y rows")
    assert_close(f64_from_bf16(dx)[rows], dyf[rows] @ wf, "sampled dx rows")
    wrows = np.sort(np.append(rng.choice(n_out, 15, replace=False), n_out - 1))
    assert_close(dw.cpu().numpy()[wrows], dyf[:, wrows].T @ xf, "sampled dW rows")


def test_split_is_bitwise_reproducible():
    """Either half of a tile may finish first; the result must not depend on which."""
    t, n_in, n_out = 4096, 4096, 28672
    inp = synth.stage_inputs("linear", 1, n_in, n_out, tokens=t, n_mb=1, seed=12)
    first = run_linear_stage(inp, t, n_in, n_out)
    for _ in range(2):
        again = run_linear_stage(inp, t, n_in, n_out)
        for a, b in zip(first, again):
            assert torch.equal(a, b)


def test_swiglu_dgrad_split_in_mlp_stage():
    """A SwiGLU-MLP layer whose down-projection dgrad (M = 4096 tokens, N = ffn 4096, K = hidden
    6144) and gate|up dgrad (N = 6144, K = 8192) split their last wave, so the SwiGLU epilogue's
    side-input ring also serves the half that only stores a partial.  dx and every gradient against
    the float64 oracle over all tokens, at the one-layer stage tolerance."""
    t, hidden, ffn = 4096, 6144, 4096
    assert _splits(t, ffn, hidden) and _splits(t, hidden, 2 * ffn)
    inp = synth.stage_inputs("mlp", 1, hidden, ffn, tokens=t, n_mb=1, seed=13)
    st = Stage.from_synth("mlp", 1, hidden, ffn, max_tokens=t, max_inflight=1, params_bits=inp["params"])
    x = bf16_from_bits(inp["x"][0])
    dy = bf16_from_bits(inp["dy"][0])
    y = torch.empty(t, hidden, dtype=torch.bfloat16, device="cuda")
    dx = torch.empty(t, hidden, dtype=torch.bfloat16, device="cuda")
    st.forward(0, x, y)
    st.backward_input(0, dy, dx)
    st.backward_weight(0)
    st.sync()
    orc = S.StageOracle(synth.params_f64(inp["params"]), dict(kind="mlp", hidden=hidden, ffn=ffn, eps=1e-5))
    orc.forward(0, synth.bf16_to_f64(inp["x"][0]))
    ref_dx = orc.backward_input(0, synth.bf16_to_f64(inp["dy"][0]))
    orc.backward_weight(0)
    tol = stage_fro_tol(1)
    assert_close(f64_from_bf16(dx), ref_dx, "dx", fro_tol=tol, max_tol=MAX_TOL)
    for k, ref in orc.grads[0].items():
        assert_close(st.grads[0][k].cpu().numpy(), ref, f"d{k}", fro_tol=tol, max_tol=MAX_TOL)
    st.close()

