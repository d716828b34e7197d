"""Comparison metrics and tolerances shared by the GPU parity tests.

Tolerances: fp32 weights and cache -> relative L2 <= 1e-4 on hidden states and
logits; bf16 weights and cache -> relative L2 <= 2e-2, cosine >= 0.999 and top-1
agreement >= 99% over all decode steps. Integer results (lengths, argmax) must
match exactly.
"""
import numpy as np

TOL_F32 = 1e-4
TOL_BF16_REL = 2e-2
TOL_BF16_COS = 0.999
TOL_TOP1 = 0.99


def rel_l2(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def cosine(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))


def top1_agreement(gpu_logits, ref_logits):
    g = np.argmax(np.asarray(gpu_logits), axis=-1)
    r = np.argmax(np.asarray(ref_logits), axis=-1)
    return float(np.mean(g == r))


def check_rows(gpu, ref, bf16, what=""):
    """Row-wise check of [rows, n] arrays against the oracle; returns the worst relative L2."""
    gpu = np.atleast_2d(np.asarray(gpu, np.float64))
    ref = np.atleast_2d(np.asarray(ref, np.float64))
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), what + ": non-finite GPU values"
    worst = max(rel_l2(g, r) for g, r in zip(gpu, ref))
    if bf16:
        assert worst <= TOL_BF16_REL, "%s: relative L2 %.3e > %.1e" % (what, worst, TOL_BF16_REL)
        wc = min(cosine(g, r) for g, r in zip(gpu, ref))
        assert wc >= TOL_BF16_COS, "%s: cosine %.6f < %.3f" % (what, wc, TOL_BF16_COS)
    else:
        assert worst <= TOL_F32, "%s: relative L2 %.3e > %.1e" % (what, worst, TOL_F32)
    return worst
