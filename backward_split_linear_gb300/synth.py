"""Seeded synthetic inputs for one pipeline stage.

This module only draws random numbers and rounds them to bf16; it holds none
of the stage's arithmetic, so both the CUDA path and the fp64 oracle can take
their inputs from it.

Recipe.  Tensors are numbered in a fixed order:
  for every layer: W_qkv, W_o, W_gu, W_down (each N(0, 0.02^2)), gamma1, gamma2
  then x for every microbatch (N(0, 1)), then dy for every microbatch (N(0, 1)).
Tensors a layer kind does not have are skipped (they take no number).  Tensor
i is filled in row-major chunks of 2^22 values; chunk j comes from numpy's
PCG64 seeded with SeedSequence(seed, spawn_key=(i, j)), so the values are the
same on every machine and the chunks can be drawn in parallel.  Weights, x and
dy are rounded to bf16 (round to nearest even); gamma stays float32 and is
either all ones or 1 + 0.1 N(0, 1).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

WEIGHT_STD = 0.02
CHUNK = 1 << 22
_THREADS = max(1, min(16, os.cpu_count() or 1))


def bf16_bits(a):
    """float32 array -> uint16 bf16 bit patterns, round to nearest even (no NaN inputs)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(bits):
    """uint16 bf16 bit patterns -> float64 values (exact)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def normal(seed, index, shape, std=1.0):
    """float32 N(0, std^2) values of tensor number `index` under `seed` (see the recipe)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)

    def fill(j):
        lo, hi = j * CHUNK, min(n, (j + 1) * CHUNK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(index, j))))
        g.standard_normal(out=out[lo:hi], dtype=np.float32)

    chunks = (n + CHUNK - 1) // CHUNK
    if chunks > 1:
        with ThreadPoolExecutor(_THREADS) as pool:
            list(pool.map(fill, range(chunks)))
    elif n:
        fill(0)
    out = out.reshape(shape)
    if std != 1.0:
        out *= np.float32(std)
    return out


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
    index = 0
    params = []
    for _ in range(n_layers):
        layer = {}
        for name, shape, is_weight in layer_param_shapes(kind, hidden, ffn, n_heads, n_kv_heads, head_dim):
            if is_weight:
                layer[name] = bf16_bits(normal(seed, index, shape, WEIGHT_STD))
            elif gamma == "ones":
                layer[name] = np.ones(shape, dtype=np.float32)
            else:
                layer[name] = (1.0 + 0.1 * normal(seed, index, shape)).astype(np.float32)
            index += 1
        params.append(layer)
    t_list = list(tokens_per_mb) if tokens_per_mb is not None else [tokens] * n_mb
    out_dim = ffn if kind == "linear" else hidden
    xs = []
    for t in t_list:
        xs.append(bf16_bits(normal(seed, index, (t, hidden))))
        index += 1
    dys = []
    for t in t_list:
        dys.append(bf16_bits(normal(seed, index, (t, out_dim))))
        index += 1
    return {"params": params, "x": xs, "dy": dys}


def params_f64(params):
    """The oracle's view: every parameter as float64."""
    out = []
    for layer in params:
        out.append({k: (bf16_to_f64(v) if v.dtype == np.uint16 else v.astype(np.float64))
                    for k, v in layer.items()})
    return out
