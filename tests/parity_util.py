"""Comparison metrics and tolerances shared by the GPU parity tests.

Tolerances: fp32 weights and cache -> relative L2 <= 1e-4 on hidden states and
logits; bf16 weights and cache -> relative L2 <= 2e-2, cosine >= 0.999 and top-1
agreement >= 99% over all decode steps. Integer results (lengths, argmax) must
match exactly.

Top-1 on near ties: a step whose oracle top-2 margin is at most twice the step's
largest logit error max_i |L_gpu[i] - L_ref[i]| is "undecided": within that error the
two leading logits may swap order, so its top-1 says nothing beyond the logits check.
Over the other ("decided") steps top-1 agreement must reach 99%; undecided steps are
counted and reported with the margin distribution.
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


def top1_decided(gpu_logits, ref_logits):
    """Top-1 agreement with the near-tie rule above. Returns a dict with the overall
    agreement, the agreement over decided steps, the number of undecided steps and the
    oracle top-2 margins (finite logits only, so suppressed entries are ignored)."""
    gpu = np.atleast_2d(np.asarray(gpu_logits, np.float64))
    ref = np.atleast_2d(np.asarray(ref_logits, np.float64))
    agree, decided, margins = [], [], []
    for gr, rr in zip(gpu, ref):
        fin = np.isfinite(rr)
        err = float(np.abs(gr[fin] - rr[fin]).max())
        top2 = np.sort(rr[fin])[-2:]
        m = float(top2[1] - top2[0])
        margins.append(m)
        decided.append(m > 2.0 * err)
        agree.append(int(np.argmax(gr)) == int(np.argmax(rr)))
    agree, decided, margins = np.array(agree), np.array(decided), np.array(margins)
    return {"agree_all": float(agree.mean()),
            "agree_decided": float(agree[decided].mean()) if decided.any() else 1.0,
            "undecided": int((~decided).sum()), "steps": int(agree.size),
            "margin_min": float(margins.min()), "margin_median": float(np.median(margins))}


def assert_top1(gpu_logits, ref_logits, what=""):
    """Top-1 >= 99% over the decided steps; prints the summary (see the module docstring)."""
    r = top1_decided(gpu_logits, ref_logits)
    print("%s top-1: %.4f over all %d steps, %.4f over decided steps, %d undecided; oracle top-2 margin "
          "min %.2e median %.2e" % (what, r["agree_all"], r["steps"], r["agree_decided"], r["undecided"],
                                     r["margin_min"], r["margin_median"]))
    assert r["undecided"] <= 0.25 * r["steps"], (what, r)
    assert r["agree_decided"] >= TOL_TOP1, (what, r)
    return r
