"""Seeded synthetic inputs for one pipeline stage.

This module only draws random numbers and rounds them to bf16; it holds none
of the stage's arithmetic, so both the CUDA path and the fp64 oracle can take
their inputs from it.

Recipe (one generator, seed fixed, draws in this order):
  for every layer: W_qkv, W_o, W_gu, W_down (each N(0, 0.02^2)), gamma1, gamma2
  then x for every microbatch (N(0, 1)), then dy for every microbatch (N(0, 1)).
Weights that a layer kind does not have are not drawn.  Weights, x and dy are
rounded to bf16 (round to nearest even); gamma stays float32 and is either all
ones or 1 + 0.1 N(0, 1).  numpy's PCG64 generator makes the draws identical on
every machine.
"""
from __future__ import annotations

import numpy as np

WEIGHT_STD = 0.02


def bf16_bits(a):
    """float32 array -> uint16 bf16 bit patterns, round to nearest even (no NaN inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    return ((u + (((u >> 16) & 1) + np.uint32(0x7FFF))) >> 16).astype(np.uint16)


def bf16_to_f64(bits):
    """uint16 bf16 bit patterns -> float64 values (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def layer_param_shapes(kind, hidden, ffn, n_heads=0, n_kv_heads=0, head_dim=0):
    """Ordered (name, shape, is_weight) of one layer's parameters; weights are [out, in]."""
    if kind == "linear":
        return [("w", (ffn, hidden), True)]
    out = []
    if kind == "transformer":
        qkv_out = (n_heads + 2 * n_kv_heads) * head_dim
        out += [("w_qkv", (qkv_out, hidden), True), ("w_o", (hidden, n_heads * head_dim), True)]
    out += [("w_gu", (2 * ffn, hidden), True), ("w_down", (hidden, ffn), True)]
    if kind == "transformer":
        out.append(("gamma1", (hidden,), False))
    out.append(("gamma2", (hidden,), False))
    return out


def stage_inputs(kind, n_layers, hidden, ffn, n_heads=0, n_kv_heads=0, head_dim=0,
                 tokens=128, n_mb=1, seed=0, gamma="perturbed", tokens_per_mb=None):
    """Draw every input of a stage run.

    Returns a dict with
      "params": list (per layer) of {name: uint16 bf16 bits (weights) or float32 (gamma)}
      "x", "dy": lists (per microbatch) of uint16 bf16 bits, shapes [T, hidden] and
                 [T, out] where out is ``ffn`` for kind "linear", else ``hidden``.
    ``tokens_per_mb`` (a list) overrides ``tokens`` per microbatch.
    """
    rng = np.random.default_rng(seed)
    params = []
    for _ in range(n_layers):
        layer = {}
        for name, shape, is_weight in layer_param_shapes(kind, hidden, ffn, n_heads, n_kv_heads, head_dim):
            if is_weight:
                layer[name] = bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(WEIGHT_STD))
            elif gamma == "ones":
                layer[name] = np.ones(shape, dtype=np.float32)
            else:
                layer[name] = (1.0 + 0.1 * rng.standard_normal(shape, dtype=np.float32)).astype(np.float32)
        params.append(layer)
    t_list = list(tokens_per_mb) if tokens_per_mb is not None else [tokens] * n_mb
    out_dim = ffn if kind == "linear" else hidden
    xs = [bf16_bits(rng.standard_normal((t, hidden), dtype=np.float32)) for t in t_list]
    dys = [bf16_bits(rng.standard_normal((t, out_dim), dtype=np.float32)) for t in t_list]
    return {"params": params, "x": xs, "dy": dys}


def params_f64(params):
    """The oracle's view: every parameter as float64."""
    out = []
    for layer in params:
        out.append({k: (bf16_to_f64(v) if v.dtype == np.uint16 else v.astype(np.float64))
                    for k, v in layer.items()})
    return out
