"""Shared helpers for the GPU parity tests: tolerances and element-wise comparison.

Tolerances (max abs error against the float64 oracle on the same inputs):
  bf16 prefill and paged decode: O <= 2e-2, LSE <= 1e-3
  FP8 prefill: O <= 6e-2 (oracle on the dequantised inputs), LSE <= 1e-3
  backward: max error <= 2e-2 of the gradient tensor's largest entry
Rows with no visible key must come back as O = 0 and LSE = -inf exactly.
"""
import json
import math
import os

import numpy as np

TOL_O_BF16 = 2e-2
TOL_LSE = 1e-3
TOL_O_FP8 = 6e-2
# backward: max |g - oracle| relative to max |oracle| per gradient tensor.  P
# and dS enter the products as bf16 (relative rounding 2^-9 per element) and
# D uses the bf16 forward output; summed over up to Nk terms of random sign
# the error stays well below 1% of the tensor's largest entry, while an index
# or sign mistake gives errors of order 1.
TOL_GRAD_REL = 2e-2


def compare_grad(name, g_gpu, g_ref, tol_rel=TOL_GRAD_REL):
    g = g_gpu.float().cpu().numpy().astype(np.float64).reshape(g_ref.shape)
    assert np.all(np.isfinite(g)), name + ": non-finite gradient"
    scale = float(np.max(np.abs(g_ref))) if g_ref.size else 0.0
    err = float(np.max(np.abs(g - g_ref))) if g.size else 0.0
    rel = err / scale if scale > 0 else err
    record(name, rel, 0.0, g.shape)
    assert rel <= tol_rel, "%s: max |g - oracle| / max |oracle| = %.3g > %.3g" % (name, rel, tol_rel)
    return rel


def f32(x):
    """The float the C ABI receives (the oracle is given exactly this value)."""
    return float(np.float32(x))


def default_scale(d):
    return f32(1.0 / math.sqrt(d))


def compare(name, o_gpu, lse_gpu, o_ref, l_ref, tol_o, tol_l):
    o = o_gpu.float().cpu().numpy().astype(np.float64).reshape(o_ref.shape)
    l = lse_gpu.float().cpu().numpy().astype(np.float64).reshape(l_ref.shape)
    empty = np.isneginf(l_ref)
    assert np.array_equal(np.isneginf(l), empty), name + ": rows without keys differ"
    assert np.all(o[empty] == 0.0), name + ": empty rows must be zero"
    assert np.all(np.isfinite(o)), name + ": non-finite output"
    e_o = float(np.max(np.abs(o - o_ref))) if o.size else 0.0
    e_l = float(np.max(np.abs(l[~empty] - l_ref[~empty]))) if (~empty).any() else 0.0
    record(name, e_o, e_l, o.shape)
    assert e_o <= tol_o, "%s: max |O - oracle| = %.3g > %.3g" % (name, e_o, tol_o)
    assert e_l <= tol_l, "%s: max |LSE - oracle| = %.3g > %.3g" % (name, e_l, tol_l)
    return e_o, e_l


def record(name, e_o, e_l, shape):
    path = os.environ.get("ATTN_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": name, "max_err_o": e_o, "max_err_lse": e_l,
                                "shape": list(shape)}) + "\n")
