"""CPU oracle for DP-SGD per-example gradient clipping.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports, calls or links this
package: only the tests, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline
and reference legs use it.  It shares no code with the CUDA path; both read their
inputs from the ``workloads`` module.

It computes the method by its plain definition, in float64 with numpy: every
per-example gradient g_i is materialised (conv layers through an explicit
im2col), its Frobenius norm taken, the clip factor formed, the clipped gradients
summed one by one, and seeded Gaussian noise added before the 1/B scale.  The
ghost-norm identity, the one-row closed form and the reweighted contraction that
the CUDA path relies on are NOT used here; the tests check them against this
definition instead.

Every function is pinned by the CPU test suite against something other than
itself (library routines such as torch autograd, torch.nn.functional.unfold and
numpy's Philox4x64, closed forms, brute force on tiny inputs, invariants of the
clip rule); see tests/test_oracle_pins.py.
"""
from .dpsgd import (  # noqa: F401
    unfold2d, unfold1d, unfold3d, per_example_grad, layer_sqnorms, clip_factors, clipped_sum,
    clipped_sum_elements,
    add_noise, adaptive_bound, norm_mode_plan, norm_mode_plan_time, dp_step, NONFINITE,
)
from .philox import philox4, normal_noise, noise_words, uniform_from_word  # noqa: F401
