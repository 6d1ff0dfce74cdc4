"""The whole-stage tolerances of the GPU tests, pinned by a bf16 replay (CPU only).

tests/parity.py holds whole stages to looser bars than single steps, because every tensor the
GPU stores is rounded to bf16 and those roundings travel down the layers.  The replay in
tests/bf16_replay.py computes a stage in float64 with exactly those roundings and nothing else
(every sum exact), so its error against the exact oracle is what bf16 storage alone costs.
Each tolerance must admit that cost, and must not exceed it by more than a small factor: a
tolerance far above what the roundings explain would hide kernel errors.  (Kernel errors are
also caught on their own, step by step at the single-step bar, by tests/test_gpu_stash_fed.py.)
"""
import numpy as np
import pytest

from backward_split_linear_gb300 import synth
from bf16_replay import replay_errors
from parity import CAUSAL_MAX_TOL, MAX_TOL, causal_stage_fro_tol, stage_fro_tol


def worst(errs):
    return max(v[0] for v in errs.values()), max(v[1] for v in errs.values())


@pytest.mark.parametrize("n_layers", [1, 2, 4])
def test_standin_stage_tolerance_grows_like_sqrt_depth(n_layers):
    """Stand-in transformer layers at reduced widths (512 / 1792, 8 / 2 heads of 64), two
    256-token microbatches: the replay's worst error over dx and every gradient lies between a
    third of 5e-3 * sqrt(4 L) and that bound, for L = 1, 2, 4."""
    c = dict(kind="transformer", n_layers=n_layers, hidden=512, ffn=1792, n_heads=8, n_kv_heads=2, head_dim=64,
             eps=1e-5, attention="standin", seq_len=0)
    inp = synth.stage_inputs("transformer", n_layers, 512, 1792, 8, 2, 64, n_mb=2, seed=23, tokens_per_mb=[256, 256])
    fro, mx = worst(replay_errors(c, inp))
    tol = stage_fro_tol(n_layers)
    assert tol / 3 <= fro <= tol, (fro, tol)
    assert mx <= MAX_TOL


def test_standin_8b_widths_two_layers():
    """Two 8B-shaped stand-in layers (4096 / 14336, 32 / 8 heads), two 256-token microbatches:
    worst error between half of the two-layer stage bound and the bound."""
    c = dict(kind="transformer", n_layers=2, hidden=4096, ffn=14336, n_heads=32, n_kv_heads=8, head_dim=128,
             eps=1e-5, attention="standin", seq_len=0)
    inp = synth.stage_inputs("transformer", 2, 4096, 14336, 32, 8, 128, n_mb=2, seed=23, tokens_per_mb=[256, 256])
    fro, mx = worst(replay_errors(c, inp))
    assert stage_fro_tol(2) / 2 <= fro <= stage_fro_tol(2), fro
    assert mx <= MAX_TOL


def test_causal_8b_widths_two_layers():
    """Two 8B-shaped layers with the causal core, two 256-token microbatches in sequences of
    128: the softmax amplifies the rounding of q and k, and the core rounds P, dS and its
    output.  The causal stage bounds (Frobenius 5e-3 * sqrt(8 L), max-abs 3e-2 * max|ref|) must
    admit the replay's worst error and stay within twice it."""
    c = dict(kind="transformer", n_layers=2, hidden=4096, ffn=14336, n_heads=32, n_kv_heads=8, head_dim=128,
             eps=1e-5, attention="causal", seq_len=128)
    inp = synth.stage_inputs("transformer", 2, 4096, 14336, 32, 8, 128, n_mb=2, seed=23, tokens_per_mb=[256, 256])
    fro, mx = worst(replay_errors(c, inp))
    assert causal_stage_fro_tol(2) / 2 <= fro <= causal_stage_fro_tol(2), fro
    assert CAUSAL_MAX_TOL / 2 <= mx <= CAUSAL_MAX_TOL, mx
    # and the replay goes past the single-step bar, which is why whole stages need their own
    assert mx > MAX_TOL * 0.9 or fro > 5e-3
