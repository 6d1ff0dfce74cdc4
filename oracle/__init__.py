"""fp64 CPU oracle for the split backward of one pipeline stage and its F/B/W orders.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline`` leg and its
``--impl reference`` arm) may import or run anything in this package.  The
library under ``backward_split_linear_gb300/`` never imports it, and this
package imports nothing from there: the two share no code.  Inputs reach both
sides from ``backward_split_linear_gb300/synth.py``, which draws seeded random
numbers and holds none of the method's arithmetic.

What it computes, and the passages it follows (page title, section):

* ``stage``: the forward pass of one stage and its backward split into B
  (input gradient) and W (weight gradient), in float64 with no intermediate
  rounding.  "Zero-Bubble Pipeline Parallelism Guide for LLMs",
  section "Core Innovation 1: Mathematical Decomposition of the Backward Pass"
  (for Y = X W the input gradient is dY times W transposed and the weight
  gradient is X transposed times dY), and section "Step-by-Step
  Implementation" (weights stored [out, in] with y = x W^T; the forward keeps
  x, B keeps dY and returns dY W, W pops both and adds dY^T x into the weight
  gradient).  The layer around the linears is a reading (pre-norm Llama layer,
  weight-free attention stand-in), listed in the module docstring.
* ``schedule``: a unit-time simulator of all p stages and the per-stage
  F/B/W orders of GPipe, 1F1B and ZB-H1 (the guide's ZB-1F1B), section
  "The Mechanics of Pipeline Bubbles" and "Core Innovation 2: The Zero-Bubble
  Scheduling Family", with the bubble closed forms of section "Mathematical
  Modeling: Bubble Fractions, Memory Bounds, and Speedups".

Pins (tests that tie this package to something other than itself) are in
``tests/test_oracle_*.py``: central finite differences, torch.autograd in
float64, the split == fused identity, the concatenated-batch identity, and the
pages' printed bubble values and diagram.  Nothing here is "parity unpinned".
"""
