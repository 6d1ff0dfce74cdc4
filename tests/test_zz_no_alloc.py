"""The gamma-gradient reduction that allocates nothing.

Some callers cannot give the library scratch memory.  They get only their
input and output tensors from a host framework, or all device memory belongs
to another allocator.  For them,
zb_op_rmsnorm_backward_gamma_noalloc keeps its partial sums in a fixed array
inside the library.  This file checks it against the caller-scratch entry
point, through the C ABI, on two calls in a row.  The file is named so that
pytest collects it last.
"""
import numpy as np
import pytest
import torch

from backward_split_linear_gb300 import binding as zb
from backward_split_linear_gb300.runtime import bf16_from_bits
from oracle import stage as S
from parity import assert_close, draw_bf16


def _case(rng, t, hidden):
    dnb, _ = draw_bf16(rng, (t, hidden))
    xb, x = draw_bf16(rng, (t, hidden), 2.0)
    _, r = S.rmsnorm(x, np.ones(hidden), 1e-5)
    rstd = torch.from_numpy(r.astype(np.float32)).cuda()
    return bf16_from_bits(dnb), bf16_from_bits(xb), rstd


@pytest.mark.gpu
def test_noalloc_matches_scratch_entry_point_twice(cuda_device):
    rng = np.random.default_rng(123)
    # Calls in a row with different sizes.  The first fills 32 x 4096 partial
    # sums of the shared array, the second only 8 x 4096: partials the first
    # call left beyond the second's range would show up if the second read
    # them.  The third is the widest row whose partition still took two parts
    # per column before the partition was capped to the array (hidden 65600).
    cases = ((4096, 4096), (64, 4096), (200, 65600))
    assert zb.zb_op_rmsnorm_backward_gamma_scratch_bytes(4096, 4096) == 32 * 4096 * 4
    assert zb.zb_op_rmsnorm_backward_gamma_scratch_bytes(64, 4096) == 8 * 4096 * 4
    for t, hidden in cases:
        dn, x, rstd = _case(rng, t, hidden)
        init = torch.from_numpy(rng.standard_normal(hidden).astype(np.float32)).cuda()
        ref = init.clone()
        nbytes = zb.zb_op_rmsnorm_backward_gamma_scratch_bytes(t, hidden)
        scratch = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
        zb.zb_op_rmsnorm_backward_gamma(dn, x, rstd, ref, t, hidden, scratch, nbytes)
        got = init.clone()
        zb.zb_op_rmsnorm_backward_gamma_noalloc(dn, x, rstd, got, t, hidden)
        torch.cuda.synchronize()
        assert_close(got.cpu().numpy(), ref.cpu().numpy(), f"noalloc dgamma, T={t}, H={hidden}")
    assert zb.zb_device_status()[0] == 0


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_its_array(cuda_device):
    cap = zb.zb_op_rmsnorm_backward_gamma_noalloc_max_floats()
    assert cap == 1 << 17
    # hidden 131072 fits (at any token count); 196608 does not
    assert zb.zb_op_rmsnorm_backward_gamma_scratch_bytes(1 << 20, 131072) <= 4 * cap
    t, hidden = 64, 196608
    # The entry point rejects exactly when the partial sums exceed its array;
    # check that on the host first, and pass full-size buffers anyway.
    assert zb.zb_op_rmsnorm_backward_gamma_scratch_bytes(t, hidden) > 4 * cap
    dn = torch.zeros(t, hidden, dtype=torch.bfloat16, device="cuda")
    rstd = torch.ones(t, dtype=torch.float32, device="cuda")
    dg = torch.zeros(hidden, dtype=torch.float32, device="cuda")
    with pytest.raises(zb.ZBError) as e:
        zb.zb_op_rmsnorm_backward_gamma_noalloc(dn, dn, rstd, dg, t, hidden)
    assert e.value.name == "ZB_ERR_SHAPE"
    torch.cuda.synchronize()
    assert torch.count_nonzero(dg).item() == 0
