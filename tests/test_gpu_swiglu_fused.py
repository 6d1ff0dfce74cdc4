"""The gate|up forward with the SwiGLU forward in its GEMM epilogue.

A stage's F computes [g | u] = n2 W_gu^T and s = silu(g) u in one CTA-pair GEMM
launch when the microbatch has at least 256 tokens and ffn is a multiple of 128
(each 256-column tile then holds 128 features of g and the same 128 of u).  The
fused launch must give the same bits as the two-launch path it replaces: the
plain GEMM (same accumulation order when K is not split) followed by the SwiGLU
row kernel (the same expression on the same bf16 g and u).  The per-step bar
against the float64 oracle is in tests/test_gpu_stash_fed.py, whose full-size
cases run the fused path with its last-wave K split.
"""
import numpy as np
import pytest
import torch

from backward_split_linear_gb300 import binding as zb
from backward_split_linear_gb300 import synth
from backward_split_linear_gb300.runtime import Stage, bf16_from_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _status_clean(cuda_device):
    zb.zb_device_status(reset=True)
    yield
    st, code = zb.zb_device_status()
    assert st == 0, f"device status word set: {code}"


@pytest.mark.parametrize("tokens,hidden,ffn", [(512, 1024, 2816), (300, 512, 1408), (256, 768, 128)])
def test_fused_forward_equals_gemm_then_row_kernel(tokens, hidden, ffn):
    inp = synth.stage_inputs("mlp", 1, hidden, ffn, tokens=tokens, n_mb=1, seed=11)
    st = Stage.from_synth("mlp", 1, hidden, ffn, max_tokens=tokens, max_inflight=1, params_bits=inp["params"])
    x = bf16_from_bits(inp["x"][0])
    y = torch.empty(tokens, hidden, dtype=torch.bfloat16, device="cuda")
    st.set_tracing(True)
    st.forward(0, x, y)
    torch.cuda.synchronize()
    trace = st.read_tracing()
    # the RMSNorm forward is the only row launch left in F: the SwiGLU went into the GEMM
    assert trace["row_forward"]["launches"] == 1
    n2 = st.stash(0, 0, "n2").clone()
    gu = st.stash(0, 0, "gu").clone()
    s = st.stash(0, 0, "s").clone()
    w_gu = st.params[0]["w_gu"]
    gu_ref = torch.full_like(gu, float("nan"))
    s_ref = torch.full_like(s, float("nan"))
    zb.zb_op_linear_forward(n2, w_gu, None, gu_ref, tokens, hidden, 2 * ffn)
    zb.zb_op_swiglu_forward(gu_ref, s_ref, tokens, ffn)
    torch.cuda.synchronize()
    assert torch.equal(gu.view(torch.int16), gu_ref.view(torch.int16)), "[g | u]"
    assert torch.equal(s.view(torch.int16), s_ref.view(torch.int16)), "s"
    st.close()


@pytest.mark.parametrize("tokens,ffn", [(200, 1024), (512, 1344)])
def test_unfused_cases_keep_two_launches(tokens, ffn):
    """Below 256 tokens (the one-CTA GEMM) or with ffn not a multiple of 128 (a 256-column
    tile would not hold g and u of the same features) the SwiGLU stays a row kernel."""
    hidden = 512
    inp = synth.stage_inputs("mlp", 1, hidden, ffn, tokens=tokens, n_mb=1, seed=12)
    st = Stage.from_synth("mlp", 1, hidden, ffn, max_tokens=tokens, max_inflight=1, params_bits=inp["params"])
    y = torch.empty(tokens, hidden, dtype=torch.bfloat16, device="cuda")
    st.set_tracing(True)
    st.forward(0, bf16_from_bits(inp["x"][0]), y)
    torch.cuda.synchronize()
    assert st.read_tracing()["row_forward"]["launches"] == 2
    gu = st.stash(0, 0, "gu").double().cpu().numpy()
    s = st.stash(0, 0, "s").double().cpu().numpy()
    g, u = gu[:, :ffn], gu[:, ffn:]
    ref = g / (1 + np.exp(-g)) * u
    assert np.max(np.abs(s - ref)) <= 2e-2 * np.max(np.abs(ref))
    st.close()
