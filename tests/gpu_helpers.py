"""Helpers shared by the GPU parity tests: tensors from the seeded problems and the
error measures the tolerances are stated in."""
import numpy as np
import torch

# Tolerances (stated for the method's floating-point paths):
#   potentials: relative L-inf error scaled by max|f|, <= 1e-4 for fp32/tf32 scores;
#   loss:       relative error <= 1e-4 (fp32/tf32), <= 2e-3 for bf16 scores.
# Only a loss bar is stated for bf16 scores; the potentials of that path are held to the
# same relative 2e-3 (the loss <a,f> + <b,g> inherits their relative error).
# The same bounds are used for transport application, Hadamard and gradient outputs
# (scaled by the largest magnitude of the oracle's output).
POT_TOL = {"fp32": 1e-4, "tf32": 1e-4, "tf32x3": 1e-4, "bf16": 2e-3}
LOSS_TOL = {"fp32": 1e-4, "tf32": 1e-4, "tf32x3": 1e-4, "bf16": 2e-3}
# Transport application, Hadamard and gradient outputs (no bound is stated for them):
# with operands rounded to the MMA type (unit roundoff u), every dot product carries an
# error of RMS u sqrt(2/(3d)) |x||y|, i.e. a relative error of 2/eps times that in each
# plan entry, plus u/sqrt(3) from rounding the weights for the second contraction; against
# a random-sign V these do not average out. For the d = 1024, eps = 0.1 workload this
# predicts a max error of ~4e-4 (tf32) and ~1.6e-3 (bf16) relative to max|P V|; the
# bounds below are 2.5x that. The fp32 path keeps 1e-4. Split tf32 splits both
# contractions (the scores' operands, and W = W_hi + W_lo, V = V_hi + V_lo in the second),
# so it is held to the fp32 bar too.
OUT_TOL = {"fp32": 1e-4, "tf32": 1e-3, "tf32x3": 1e-4, "bf16": 4e-3}
# The single-CTA tf32 kernels (FLASHOT_WSUM_PAIRS=0) split only the score operands: their
# second contraction is single tf32, held to the tf32 bar.
OUT_TOL_SINGLE_CTA = {"fp32": 1e-4, "tf32": 1e-3, "tf32x3": 1e-3, "bf16": 4e-3}


def to_dev(arr):
    return None if arr is None else torch.from_numpy(np.ascontiguousarray(arr)).cuda()


def problem_tensors(pr, uniform_as_none=True):
    X = to_dev(pr.X)
    Y = to_dev(pr.Y)
    a = None if (uniform_as_none and pr.uniform_weights) else to_dev(pr.a)
    b = None if (uniform_as_none and pr.uniform_weights) else to_dev(pr.b)
    return X, Y, a, b


def scaled_linf(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = max(np.abs(ref).max(), 1e-30)
    return float(np.abs(got - ref).max() / scale)


def rel_err(got, ref):
    return abs(float(got) - float(ref)) / max(abs(float(ref)), 1e-30)


def pot_err(f, g, f_ref, g_ref):
    """Relative L-inf error of the potential pair, scaled by the largest potential
    magnitude of the reference: max(|f - f_ref|, |g - g_ref|) / max(|f_ref|, |g_ref|).
    (f, g) are defined jointly, so one scale serves both."""
    f, g, f_ref, g_ref = (np.asarray(x, np.float64) for x in (f, g, f_ref, g_ref))
    scale = max(np.abs(f_ref).max(), np.abs(g_ref).max(), 1e-30)
    return float(max(np.abs(f - f_ref).max(), np.abs(g - g_ref).max()) / scale)


# Unit roundoff of the score contraction's operands (round to nearest): tf32 2^-11, bf16
# 2^-9 (relative error of one rounded operand). For fp32 and split tf32 (hi.hi + hi.lo +
# lo.hi, dropped terms ~2^-22) the bound is set by fp32 accumulation over up to ~3d terms,
# taken as 2^-20.
OPERAND_U = {"fp32": 2.0 ** -20, "tf32": 2.0 ** -11, "tf32x3": 2.0 ** -20, "bf16": 2.0 ** -9}
# Rounding of the second contraction's operands (plan weights and V) in apply / gradient:
# split tf32 rounds only W_lo = W - tf32(W) (to bf16) and drops W_lo V_lo, ~2^-20 of W.
SECOND_U = {"fp32": 2.0 ** -24, "tf32": 2.0 ** -11, "tf32x3": 2.0 ** -20, "bf16": 2.0 ** -9}


def half_step_bound(precision, P, Q, eps, ref):
    """Rigorous worst case of one half-step's error from rounding the operands of <p, q>:
    each dot moves by at most 2u sum_k |p_k q_k|, each score by 2/eps times that, and the
    soft-min f = -eps log sum ... by at most eps times the largest score error, so
    |df_i| <= 4u max_j sum_k |p_ik||q_jk|. Plus the fp32 epilogue (1e-6 relative)."""
    P = np.abs(np.asarray(P, np.float64))
    Q = np.abs(np.asarray(Q, np.float64))
    worst = (P @ Q.T).max(axis=1)
    return 4.0 * OPERAND_U[precision] * worst + 1e-6 * np.abs(ref).max()
