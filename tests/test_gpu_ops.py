"""GPU parity of every per-step operation against the float64 oracle (seeded inputs).

Shapes span several 128 x 256 output tiles and leave ragged tails in every
dimension the kernels tile (tokens, output features, contraction length).
Bar: relative Frobenius <= 5e-3 and max-abs <= 2e-2 * max|ref| (tests/parity.py).
"""
import numpy as np
import pytest
import torch

from backward_split_linear_gb300 import binding as zb
from backward_split_linear_gb300.runtime import bf16_from_bits, f64_from_bf16
from oracle import stage as S
from parity import assert_close, draw_bf16

pytestmark = pytest.mark.gpu

LIN = {"kind": "linear"}


def empty_bf16(*shape):
    return torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")


def f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


@pytest.fixture(autouse=True)
def _status_clean(cuda_device):
    zb.zb_device_status(reset=True)
    yield
    st, code = zb.zb_device_status()
    assert st == 0, f"device status word set: {code}"


GEMM_SHAPES = [(1, 64, 64), (127, 320, 576), (421, 256, 832), (300, 512, 256), (1000, 128, 64)]


@pytest.mark.parametrize("t,n_in,n_out", GEMM_SHAPES)
@pytest.mark.parametrize("residual", [False, True])
def test_linear_forward(t, n_in, n_out, residual):
    rng = np.random.default_rng(10 + t)
    xb, x = draw_bf16(rng, (t, n_in))
    wb, w = draw_bf16(rng, (n_out, n_in), 0.05)
    rb, r = draw_bf16(rng, (t, n_out))
    y = empty_bf16(t, n_out)
    zb.zb_op_linear_forward(bf16_from_bits(xb), bf16_from_bits(wb), bf16_from_bits(rb) if residual else None,
                            y, t, n_in, n_out)
    ref, _ = S.layer_forward(x, {"w": w}, LIN)
    if residual:
        ref = ref + r
    assert_close(f64_from_bf16(y), ref, "linear forward")


@pytest.mark.parametrize("t,n_in,n_out", GEMM_SHAPES)
def test_backward_input(t, n_in, n_out):
    rng = np.random.default_rng(20 + t)
    dyb, dy = draw_bf16(rng, (t, n_out))
    wb, w = draw_bf16(rng, (n_out, n_in), 0.05)
    dx = empty_bf16(t, n_in)
    zb.zb_op_backward_input(bf16_from_bits(dyb), bf16_from_bits(wb), dx, t, n_in, n_out)
    ref, _ = S.layer_backward_input(dy, {"w": w}, None, LIN)
    assert_close(f64_from_bf16(dx), ref, "backward input")


@pytest.mark.parametrize("t_list,n_in,n_out", [((421, 77), 320, 576), ((1, 1000), 256, 832),
                                               ((128, 256), 64, 64), ((0, 333), 128, 384)])
def test_backward_weight_accumulates(t_list, n_in, n_out):
    rng = np.random.default_rng(30 + n_out)
    acc0 = rng.standard_normal((n_out, n_in)).astype(np.float32)
    dw = f32(acc0)
    ref = {"w": acc0.astype(np.float64)}
    for t in t_list:
        xb, x = draw_bf16(rng, (t, n_in))
        dyb, dy = draw_bf16(rng, (t, n_out))
        zb.zb_op_backward_weight(bf16_from_bits(dyb), bf16_from_bits(xb), dw, t, n_in, n_out)
        S.layer_backward_weight(ref, {"x": x}, {"dy": dy}, LIN)
    assert_close(dw.cpu().numpy(), ref["w"], "backward weight")


@pytest.mark.parametrize("shapes", [[(512, 768), (320, 1024), (1024, 256), (640, 640)],
                                    [(256, 512), (64, 128), (512, 256)]])
def test_backward_weight_group_equals_separate_calls(shapes):
    """One grouped W launch gives the same bits as one call per linear (onto non-zero
    accumulators); the second case has an output too small for the CTA-pair kernel, so the
    group runs as separate launches."""
    t = 700
    rng = np.random.default_rng(77)
    dys, xs, acc0 = [], [], []
    for n_in, n_out in shapes:
        dys.append(bf16_from_bits(draw_bf16(rng, (t, n_out))[0]))
        xs.append(bf16_from_bits(draw_bf16(rng, (t, n_in))[0]))
        acc0.append(f32(rng.standard_normal((n_out, n_in))))
    grouped = [a.clone() for a in acc0]
    zb.zb_op_backward_weight_group(dys, xs, grouped, t, [s[0] for s in shapes], [s[1] for s in shapes])
    for i, (n_in, n_out) in enumerate(shapes):
        single = acc0[i].clone()
        zb.zb_op_backward_weight(dys[i], xs[i], single, t, n_in, n_out)
        assert torch.equal(grouped[i], single), shapes[i]
        ref = acc0[i].double().cpu().numpy() + (f64_from_bf16(dys[i]).T @ f64_from_bf16(xs[i]))
        assert_close(grouped[i].cpu().numpy(), ref, f"grouped dW {shapes[i]}")


def test_backward_weight_bitwise_reproducible():
    rng = np.random.default_rng(5)
    xb, _ = draw_bf16(rng, (777, 384))
    dyb, _ = draw_bf16(rng, (777, 640))
    out = []
    for _ in range(2):
        dw = torch.zeros(640, 384, dtype=torch.float32, device="cuda")
        for _ in range(3):
            zb.zb_op_backward_weight(bf16_from_bits(dyb), bf16_from_bits(xb), dw, 777, 384, 640)
        out.append(dw.cpu())
    assert torch.equal(out[0], out[1])


@pytest.mark.parametrize("t,hidden,ffn", [(300, 256, 576), (128, 256, 1024), (1, 64, 64)])
@pytest.mark.parametrize("in_place", [False, True])
def test_backward_input_swiglu(t, hidden, ffn, in_place):
    rng = np.random.default_rng(40 + t)
    dyb, dy = draw_bf16(rng, (t, hidden))
    wb, w = draw_bf16(rng, (hidden, ffn), 0.02)
    gub, gu = draw_bf16(rng, (t, 2 * ffn), 1.3)
    gu_dev = bf16_from_bits(gub)
    dgu = gu_dev if in_place else empty_bf16(t, 2 * ffn)
    zb.zb_op_backward_input_swiglu(bf16_from_bits(dyb), bf16_from_bits(wb), gu_dev, dgu, t, hidden, ffn)
    dg, du = S.swiglu_grads(dy @ w, gu[:, :ffn], gu[:, ffn:])
    got = f64_from_bf16(dgu)
    assert_close(got[:, :ffn], dg, "dg")
    assert_close(got[:, ffn:], du, "du")


@pytest.mark.parametrize("t,hidden,n_out", [(300, 256, 1152), (129, 512, 768), (1, 64, 192)])
def test_backward_input_rmsnorm(t, hidden, n_out):
    rng = np.random.default_rng(50 + t)
    dyb, dy = draw_bf16(rng, (t, n_out))
    wb, w = draw_bf16(rng, (n_out, hidden), 0.02)
    xb, x = draw_bf16(rng, (t, hidden), 2.0)
    drb, dres = draw_bf16(rng, (t, hidden))
    gamma = (1.0 + 0.1 * rng.standard_normal(hidden)).astype(np.float32)
    _, r = S.rmsnorm(x, gamma.astype(np.float64), 1e-5)
    r32 = r.astype(np.float32)
    dn = empty_bf16(t, hidden)
    dx = empty_bf16(t, hidden)
    zb.zb_op_backward_input_rmsnorm(bf16_from_bits(dyb), bf16_from_bits(wb), bf16_from_bits(xb), f32(r32),
                                    f32(gamma), bf16_from_bits(drb), dn, dx, t, hidden, n_out)
    dn_ref = dy @ w
    dx_ref = dres + S.rmsnorm_input_grad(dn_ref, x, r32.astype(np.float64), gamma.astype(np.float64))
    assert_close(f64_from_bf16(dn), dn_ref, "dn")
    assert_close(f64_from_bf16(dx), dx_ref, "dx")


@pytest.mark.parametrize("t,nh,nkv,hd", [(300, 4, 2, 64), (77, 8, 1, 64), (128, 4, 4, 32)])
def test_backward_input_attention(t, nh, nkv, hd):
    rng = np.random.default_rng(60 + t)
    h = nh * hd
    dhb, dh = draw_bf16(rng, (t, h))
    wb, w = draw_bf16(rng, (h, h), 0.02)
    dqkv = empty_bf16(t, (nh + 2 * nkv) * hd)
    zb.zb_op_backward_input_attention(bf16_from_bits(dhb), bf16_from_bits(wb), dqkv, t, nh, nkv, hd)
    ref = S.attention_standin_grad(dh @ w, nh, nkv, hd)
    assert_close(f64_from_bf16(dqkv), ref, "dqkv")


@pytest.mark.parametrize("t,hidden", [(1000, 256), (33, 512), (4096, 64), (1, 128)])
def test_rmsnorm_backward_gamma(t, hidden):
    rng = np.random.default_rng(70 + t)
    dnb, dn = draw_bf16(rng, (t, hidden))
    xb, x = draw_bf16(rng, (t, hidden), 2.0)
    _, r = S.rmsnorm(x, np.ones(hidden), 1e-5)
    r32 = r.astype(np.float32)
    init = rng.standard_normal(hidden).astype(np.float32)
    dg = f32(init)
    nbytes = zb.zb_op_rmsnorm_backward_gamma_scratch_bytes(t, hidden)
    scratch = torch.empty(nbytes // 4 + 4, dtype=torch.float32, device="cuda")
    for _ in range(2):
        zb.zb_op_rmsnorm_backward_gamma(bf16_from_bits(dnb), bf16_from_bits(xb), f32(r32), dg, t, hidden,
                                        scratch, nbytes)
    ref = init + 2 * S.rmsnorm_gamma_grad(dn, x, r32.astype(np.float64))
    assert_close(dg.cpu().numpy(), ref, "dgamma")


@pytest.mark.parametrize("t,hidden", [(300, 256), (5, 8192), (64, 320)])
def test_rmsnorm_forward(t, hidden):
    rng = np.random.default_rng(80 + t)
    xb, x = draw_bf16(rng, (t, hidden), 3.0)
    gamma = (1.0 + 0.1 * rng.standard_normal(hidden)).astype(np.float32)
    n = empty_bf16(t, hidden)
    rstd = torch.empty(t, dtype=torch.float32, device="cuda")
    zb.zb_op_rmsnorm_forward(bf16_from_bits(xb), f32(gamma), 1e-5, n, rstd, t, hidden)
    n_ref, r_ref = S.rmsnorm(x, gamma.astype(np.float64), 1e-5)
    assert_close(f64_from_bf16(n), n_ref, "n")
    assert_close(rstd.cpu().numpy(), r_ref, "rstd", fro_tol=1e-5, max_tol=1e-5)


def test_swiglu_and_attention_forward():
    rng = np.random.default_rng(90)
    t, ffn = 200, 320
    gub, gu = draw_bf16(rng, (t, 2 * ffn), 1.3)
    s = empty_bf16(t, ffn)
    zb.zb_op_swiglu_forward(bf16_from_bits(gub), s, t, ffn)
    assert_close(f64_from_bf16(s), S.silu(gu[:, :ffn]) * gu[:, ffn:], "swiglu")
    nh, nkv, hd = 8, 2, 64
    qb, q = draw_bf16(rng, (t, (nh + 2 * nkv) * hd))
    a = empty_bf16(t, nh * hd)
    zb.zb_op_attention_forward(bf16_from_bits(qb), a, t, nh, nkv, hd)
    assert_close(f64_from_bf16(a), S.attention_standin(q, nh, nkv, hd), "attention stand-in")


def test_zero_tokens_is_a_no_op():
    dw = torch.ones(64, 64, dtype=torch.float32, device="cuda")
    dummy = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    zb.zb_op_backward_weight(dummy, dummy, dw, 0, 64, 64)
    zb.zb_op_backward_input(dummy, dummy, dummy, 0, 64, 64)
    torch.cuda.synchronize()
    assert torch.equal(dw, torch.ones_like(dw))


def test_wait_timeout_is_reported_and_cleared():
    """A wait on a barrier nothing arrives on gives up, sets the status word, and the context stays usable."""
    zb.zb_selftest_wait_timeout(2000)
    st, code = zb.zb_device_status(reset=True)
    assert st == -7 and code == 9
    assert zb.zb_device_status()[0] == 0
    test_backward_input(127, 320, 576)


@pytest.mark.parametrize("t,n_in,n_out", [(4096, 4096, 512), (4000, 4032, 320)])
def test_backward_input_many_tiles(t, n_in, n_out):
    """256 CTA-pair tiles, 3.4 waves of 76 pairs, with the TMA-store epilogue (ragged M and N in the
    second case); per-step ops never split K."""
    rng = np.random.default_rng(21)
    dyb, dy = draw_bf16(rng, (t, n_out))
    wb, w = draw_bf16(rng, (n_out, n_in), 0.05)
    dx = empty_bf16(t, n_in)
    zb.zb_op_backward_input(bf16_from_bits(dyb), bf16_from_bits(wb), dx, t, n_in, n_out)
    assert_close(f64_from_bf16(dx), dy @ w, "backward input, many tiles")


@pytest.mark.parametrize("residual", [False, True])
def test_narrow_last_wave_same_bits(residual):
    """On 76 CTA pairs, 4096 x 4096 outputs leave a last wave of 28 of 256 tiles, which the GEMM
    runs as 56 units of 256 x 128; 4352 rows (272 tiles, 44 left over) keep whole tiles.  Every
    output element takes the same K steps in both, so the first 4096 rows agree bit for bit;
    both against the float64 product on sampled rows."""
    n_in, n_out = 512, 4096
    rng = np.random.default_rng(24)
    xb, x = draw_bf16(rng, (4352, n_in))
    wb, w = draw_bf16(rng, (n_out, n_in), 0.05)
    rb, r = draw_bf16(rng, (4352, n_out))
    ys = []
    for t in (4096, 4352):
        y = empty_bf16(t, n_out)
        zb.zb_op_linear_forward(bf16_from_bits(xb[:t]), bf16_from_bits(wb), bf16_from_bits(rb[:t]) if residual else None,
                                y, t, n_in, n_out)
        ys.append(y)
    torch.cuda.synchronize()
    assert torch.equal(ys[0], ys[1][:4096])
    rows = np.sort(np.append(rng.choice(4096, 31, replace=False), 4095))
    ref = x[rows] @ w.T + (r[rows] if residual else 0.0)
    assert_close(f64_from_bf16(ys[0])[rows], ref, "narrow last wave, sampled rows")


@pytest.mark.parametrize("t,n_in,n_out", [(300, 4096, 4096), (129, 4032, 4000 // 64 * 64)])
def test_backward_weight_many_tiles(t, n_in, n_out):
    rng = np.random.default_rng(22)
    xb, x = draw_bf16(rng, (t, n_in))
    dyb, dy = draw_bf16(rng, (t, n_out))
    dw = torch.zeros(n_out, n_in, dtype=torch.float32, device="cuda")
    zb.zb_op_backward_weight(bf16_from_bits(dyb), bf16_from_bits(xb), dw, t, n_in, n_out)
    assert_close(dw.cpu().numpy(), dy.T @ x, "backward weight, many tiles")


def test_backward_input_swiglu_many_tiles():
    rng = np.random.default_rng(23)
    t, hidden, ffn = 4096, 256, 4096
    dyb, dy = draw_bf16(rng, (t, hidden))
    wb, w = draw_bf16(rng, (hidden, ffn), 0.05)
    gub, gu = draw_bf16(rng, (t, 2 * ffn), 1.3)
    dgu = empty_bf16(t, 2 * ffn)
    zb.zb_op_backward_input_swiglu(bf16_from_bits(dyb), bf16_from_bits(wb), bf16_from_bits(gub), dgu, t, hidden, ffn)
    dg, du = S.swiglu_grads(dy @ w, gu[:, :ffn], gu[:, ffn:])
    got = f64_from_bf16(dgu)
    assert_close(got[:, :ffn], dg, "dg, many tiles")
    assert_close(got[:, ffn:], du, "du, many tiles")
