"""libzb checks that need no GPU: exports, the schedule generator, host-side argument checks."""
import ctypes
import os
import re

import pytest

from backward_split_linear_gb300 import binding as zb
from oracle import schedule as S

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "zb.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zb_\w+)\s*\(", text)))


def test_exports_every_declared_function(zblib):
    names = header_functions()
    assert len(names) >= 25
    for name in names:
        assert hasattr(zblib, name), name
    assert sorted(zb.declared_symbols()) == names


def test_device_status_codes_documented():
    """The device status codes that zb.h lists are the kernels' wait sites, code for code."""
    src = open(os.path.join(os.path.dirname(HEADER), "..", "backward_split_linear_gb300", "csrc",
                            "device_common.cuh")).read()
    enum = src[src.index("enum WaitSite"):src.index("};", src.index("enum WaitSite"))]
    sites = {int(v) for v in re.findall(r"kSite\w+\s*=\s*(\d+)", enum)}
    text = open(HEADER).read()
    start = text.index("Device status word")
    block = text[start:text.index("zb_device_status(", start)]
    listed = {int(v) for v in re.findall(r"^\s*\*\s+(\d+)\s+\S", block, flags=re.M)}
    assert sites == set(range(1, max(sites) + 1))
    assert listed == sites


def test_version_and_status_strings(zblib):
    assert zb.zb_version() == 100
    for code in zb.STATUS_NAMES:
        assert zb.zb_status_string(code) != "unknown status"


@pytest.mark.parametrize("kind", ["1f1b", "zbh1", "gpipe", "zb2p"])
def test_generator_equals_oracle(zblib, kind):
    """The library's orders equal the oracle's simulator, op for op."""
    for p in range(1, 13):
        for m in list(range(1, 3 * p + 2)) + [40]:
            ref = S.orders_for(kind, p, m)
            for s in range(p):
                assert zb.zb_schedule(kind, s, p, m) == ref[s], (kind, s, p, m)


def test_zbh1_stage3_p8_m16_order(zblib):
    """ZB-H1 for stage 3 of p = 8, m = 16: W deferred behind B, steady B W F rhythm, drain at the end."""
    got = " ".join(f"{k}{i}" for k, i in zb.zb_schedule("zbh1", 3, 8, 16))
    want = ("F0 F1 F2 F3 F4 B0 F5 B1 F6 B2 F7 B3 W0 F8 B4 W1 F9 B5 W2 F10 B6 W3 F11 B7 W4 F12 "
            "B8 W5 F13 B9 W6 F14 B10 W7 F15 B11 W8 B12 W9 B13 W10 B14 W11 B15 W12 W13 W14 W15")
    assert got == want


@pytest.mark.parametrize("kind", ["1f1b", "zbh1", "gpipe", "zb2p"])
@pytest.mark.parametrize("p,m", [(1, 1), (2, 5), (4, 3), (8, 16), (8, 12), (8, 24), (8, 32), (6, 40)])
def test_bubble_model_equals_oracle(zblib, kind, p, m):
    span, over_c, over_w = zb.zb_schedule_bubble(kind, p, m)
    c, w = S.bubble(kind, p, m)
    _, start = S.timeline(kind, p, m)
    assert span == S.makespan(start)
    assert abs(over_c - c) < 1e-12 and abs(over_w - w) < 1e-12
    units, frac = zb.zb_schedule_window_idle(kind, p, m)
    assert units == S.window_idle(kind, p, m)
    assert abs(frac - units / (3 * m * p)) < 1e-15


def test_bubble_printed_values(zblib):
    # "Zero-Bubble Pipeline Parallelism Guide for LLMs": 7/16 (section "2. The 1F1B ..."),
    # 30.4 % of wall time (first diagram), (p-1)/(3m) for ZB-1F1B (section "Mathematical Modeling")
    assert abs(zb.zb_schedule_bubble("1f1b", 8, 16)[1] - 7 / 16) < 1e-12
    assert round(100 * zb.zb_schedule_bubble("1f1b", 8, 16)[2], 1) == 30.4
    assert abs(zb.zb_schedule_bubble("zbh1", 8, 16)[1] - 7 / 48) < 1e-12


def test_schedule_errors(zblib):
    st, n, _ = zb.zb_schedule_raw(1, 0, 4, 8, 10)
    assert st == -8 and n == 24  # ZB_ERR_CAPACITY reports the size needed
    assert zb.zb_schedule_raw(1, 4, 4, 8, 24)[0] == -1  # stage out of range
    assert zb.zb_schedule_raw(1, 0, 0, 8, 24)[0] == -1
    assert zb.zb_schedule_raw(1, 0, 4, 0, 24)[0] == -1
    assert zb.zb_schedule_raw(7, 0, 4, 8, 24)[0] == -1  # unknown kind
    assert zb.zb_schedule_window_idle("zb2p", 8, 16) == (0, 0.0)
    assert zb.zb_schedule_raw(1, 0, 4, 8, 24)[0] == 0


def test_stage_config_checks(zblib):
    ok = zb.make_config("transformer", 2, 256, 512, 4, 2, 64, max_tokens=128, max_inflight=2)
    assert zb.zb_stage_workspace_bytes(ok) > 0
    bad_shape = zb.make_config("transformer", 2, 256, 500, 4, 2, 64)   # ffn not a multiple of 64
    assert zb.zb_stage_workspace_bytes(bad_shape) == 0
    bad_heads = zb.make_config("transformer", 2, 256, 512, 4, 3, 64)   # 4 heads, 3 kv heads
    assert zb.zb_stage_workspace_bytes(bad_heads) == 0
    bad_linear = zb.make_config("linear", 2, 256, 512)                 # a linear stage has one layer
    assert zb.zb_stage_workspace_bytes(bad_linear) == 0
    # every stash slot adds one microbatch's stash: per MLP layer x, n2, dy, dn2 [T, H],
    # [g|u] [T, 2F], s [T, F] in bf16 and rstd [T] in float32
    T, H, F, L = 128, 256, 1024, 2
    per_slot = L * (4 * T * H * 2 + T * 2 * F * 2 + T * F * 2 + T * 4)
    one = zb.zb_stage_workspace_bytes(zb.make_config("mlp", L, H, F, max_tokens=T, max_inflight=1))
    four = zb.zb_stage_workspace_bytes(zb.make_config("mlp", L, H, F, max_tokens=T, max_inflight=4))
    assert one >= per_slot
    assert four - one >= 3 * per_slot
    scratch = zb.zb_op_rmsnorm_backward_gamma_scratch_bytes(128, 256)
    assert scratch > 0 and scratch % (256 * 4) == 0  # whole float32 rows of partial sums


def test_stage_host_errors_without_device(zblib):
    """Creation and order errors are decided on the host, before any device call."""
    cfg = zb.make_config("linear", 1, 256, 512, max_tokens=64, max_inflight=1)
    nbytes = zb.zb_stage_workspace_bytes(cfg)
    fake = 1 << 20  # never dereferenced by these calls
    with pytest.raises(zb.ZBError) as e:
        zb.zb_stage_create(cfg, [{"w": fake, "dw": fake}], fake + 8, nbytes)
    assert e.value.name == "ZB_ERR_WORKSPACE"  # misaligned workspace
    with pytest.raises(zb.ZBError) as e:
        zb.zb_stage_create(cfg, [{"w": fake}], fake, nbytes)
    assert e.value.name == "ZB_ERR_ARG"  # missing accumulator
    st = zb.zb_stage_create(cfg, [{"w": fake, "dw": fake}], fake, nbytes)
    try:
        with pytest.raises(zb.ZBError) as e:
            zb.zb_backward_input(st, 0, fake, fake, 0)
        assert e.value.name == "ZB_ERR_NO_MB"
        with pytest.raises(zb.ZBError) as e:
            zb.zb_backward_weight(st, 3, 0)
        assert e.value.name == "ZB_ERR_NO_MB"
        with pytest.raises(zb.ZBError) as e:
            zb.zb_stage_forward(st, 0, fake, 65, fake, 0)
        assert e.value.name == "ZB_ERR_SHAPE"  # tokens > max_tokens
        assert zb.zb_stage_stats(st) == (0, 0, 0)
        zb.zb_wgrad_flush(st, 0)  # nothing pending: no device call
        # the stash view of a microbatch that is not in flight, or of a bad layer or tensor
        with pytest.raises(zb.ZBError) as e:
            zb.zb_stage_stash_view(st, 0, 0, "x")
        assert e.value.name == "ZB_ERR_NO_MB"
        for layer, tensor in ((1, "x"), (-1, "x"), (0, len(zb.STASH_TENSORS))):
            with pytest.raises(zb.ZBError) as e:
                zb.zb_stage_stash_view(st, 0, layer, tensor)
            assert e.value.name == "ZB_ERR_ARG"
    finally:
        zb.zb_stage_destroy(st)


def test_op_argument_errors(zblib):
    fake = 1 << 20
    lib = zblib
    assert lib.zb_op_backward_weight(None, fake, fake, 8, 64, 64, None) == -1
    assert lib.zb_op_backward_weight(fake + 2, fake, fake, 8, 64, 64, None) == -1  # misaligned
    assert lib.zb_op_backward_weight(fake, fake, fake, 8, 65, 64, None) == -2
    assert lib.zb_op_backward_weight(fake, fake, fake, -1, 64, 64, None) == -2
    assert lib.zb_op_backward_input_attention(fake, fake, fake, 8, 6, 4, 64, None) == -2  # 4 does not divide 6
    assert lib.zb_op_rmsnorm_backward_gamma(fake, fake, fake, fake, 64, 256, fake, 10, None) == -10


def test_causal_attention_host_checks(zblib):
    """Shape rules of the causal attention core, decided on the host before any device call."""
    assert zb.zb_op_attention_stat_stride(0) == 128
    assert zb.zb_op_attention_stat_stride(129) == 256
    fake = 1 << 20  # never dereferenced: the calls below fail their shape checks first
    for nh, nkv, d, seq_len in [(4, 2, 96, 0), (4, 2, 64, 100), (4, 3, 64, 0), (4, 2, 64, -128)]:
        with pytest.raises(zb.ZBError) as e:
            zb.zb_op_attention_causal_forward(fake, fake, fake, 256, nh, nkv, d, seq_len, stream=0)
        assert e.value.name == "ZB_ERR_SHAPE"
        with pytest.raises(zb.ZBError) as e:
            zb.zb_op_attention_causal_backward(fake, fake, fake, fake, fake, fake, 256, nh, nkv, d, seq_len,
                                               stream=0)
        assert e.value.name == "ZB_ERR_SHAPE"
    tf = dict(kind="transformer", n_layers=2, hidden=256, ffn=512, n_heads=4, n_kv_heads=2, head_dim=64,
              max_tokens=256, max_inflight=2)
    standin = zb.zb_stage_workspace_bytes(zb.make_config(**tf))
    causal = zb.zb_stage_workspace_bytes(zb.make_config(**tf, attention="causal", seq_len=128))
    # the causal stash adds qkv [T, 512] bf16 and lse [4, 256] float32 per layer and slot
    assert causal - standin >= 2 * 2 * (256 * 512 * 2 + 4 * 256 * 4) - 256 * 512 * 2
    assert zb.zb_stage_workspace_bytes(zb.make_config(**tf, attention="causal", seq_len=100)) == 0
    assert zb.zb_stage_workspace_bytes(zb.make_config(**tf, seq_len=128)) == 0  # stand-in has no sequences
    assert zb.zb_stage_workspace_bytes(zb.make_config("mlp", 2, 256, 512, max_tokens=128,
                                                      attention="causal")) == 0


def test_schedule_search_equals_oracle(zblib):
    """The library's memory-limited search gives the oracle's order, ceiling and makespan."""
    from oracle import schedule as OS

    for p, m in [(1, 3), (2, 5), (4, 8), (4, 13), (8, 16)]:
        for mem in (p, p + p // 2, 2 * p, 3 * p):
            for tf, tb, tw in [(1, 1, 1), (10, 12, 9), (3, 7, 2), (5, 5, 11)]:
                limit, span, orders = OS.search_limit(p, m, mem, tf, tb, tw)
                for s in range(p):
                    got = zb.zb_schedule_search(s, p, m, mem, tf, tb, tw)
                    assert got == (orders[s], limit, span), (p, m, mem, tf, tb, tw, s)
    with pytest.raises(zb.ZBError) as e:
        zb.zb_schedule_search(0, 4, 8, 3, 1, 1, 1)  # a ceiling below p cannot hold the warm-up
    assert e.value.name == "ZB_ERR_ARG"


def test_noalloc_size_rule_holds_for_every_width(zblib):
    """zb.h promises that the allocation-free gamma reduction takes every token count for
    hidden <= 131072: its partial sums (zb_op_rmsnorm_backward_gamma_scratch_bytes) must
    fit the library's fixed array for each multiple of 64 up to there, at any T."""
    from backward_split_linear_gb300 import binding as zb

    cap = 4 * zb.zb_op_rmsnorm_backward_gamma_noalloc_max_floats()
    assert cap == 512 * 1024
    for hidden in range(64, 131072 + 1, 64):
        for t in (1, 8, 9, 63, 1000, 4096, 1 << 20, 1 << 24):
            nbytes = zb.zb_op_rmsnorm_backward_gamma_scratch_bytes(t, hidden)
            assert 0 < nbytes <= cap, (t, hidden, nbytes)
    # past the promise the partition needs more than the array for long inputs
    assert zb.zb_op_rmsnorm_backward_gamma_scratch_bytes(1 << 20, 131072 + 64) > cap


def test_stash_tensor_names_follow_the_header():
    """binding.STASH_TENSORS is the zb_stash_tensor enum of include/zb.h, in order."""
    import re

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "include", "zb.h")) as fh:
        text = fh.read()
    body = text[text.index("typedef enum {\n    ZB_STASH_X"):text.index("} zb_stash_tensor;")]
    names = [n.lower() for n in re.findall(r"ZB_STASH_([A-Z0-9]+)", body) if n != "COUNT"]
    assert names == zb.STASH_TENSORS


def test_kernel_class_names_follow_the_header():
    """binding.KERNEL_CLASSES is the zb_kernel_class enum of include/zb.h, in order."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "include", "zb.h")) as fh:
        text = fh.read()
    body = text[text.index("    ZB_KCLASS_GEMM_FORWARD = 0"):text.index("} zb_kernel_class;")]
    names = [n.lower() for n in re.findall(r"ZB_KCLASS_([A-Z_]+)", body) if n != "COUNT"]
    assert names == zb.KERNEL_CLASSES
