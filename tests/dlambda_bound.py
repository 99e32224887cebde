"""Tolerance of the lambda gradient, and the check that it can still fail.

dlambda = sum_i t_i over every query row i, with t_i = -<g_i, A2 V_i>, where
g_i is the gradient of the loss with respect to row i's pre-norm output
(through the GroupNorm and gain).  The kernels build each t_i from two
forward outputs: the pre-norm output (which g_i depends on through the
GroupNorm statistics) and A2 V.  Both carry the forward's rounding of the
probabilities to bf16 before the P V product, a relative error uniform in
[-2^-9, 2^-9] per probability, i.e. RMS 2^-9 / sqrt(3) = 1.13e-3 relative
on each output (the normalisation by the sum of the same rounded values
keeps it relative, whatever the number of keys).  Each term therefore
carries two independent errors of RMS 1.13e-3 |t_i|, RMS sqrt(2) * 1.13e-3
|t_i| = 1.59e-3 |t_i| in all, and the rows' errors are independent, so the
error of the sum has RMS 1.59e-3 * rss, rss = sqrt(sum_i t_i^2) (the oracle
reports it as dlambda_rss).  The bound allows two standard deviations of
that, 2 sqrt(2/3) 2^-9 = 3.19e-3 ~ 3e-3, on top of 1e-2 of |dlambda| for the
fp32 accumulation over rows.

A bound of this size is only useful if it still rejects the mistakes a
kernel could make in dlambda.  `assert_rejects_plausible_bugs` checks, for
the values of the case at hand, that it rejects an error the size of one
row's typical term (a wrong or dropped subset of rows, o_pre used in place
of A2 V) and, unless dlambda cancels to far below its terms, a flipped sign
or a dropped lambda term (GPU value -dlambda or 0).
"""
import math

KAPPA = 2.0 * math.sqrt(2.0 / 3.0) * 2.0 ** -9   # 3.19e-3
REL = 1e-2


def bound(ref: float, rss: float) -> float:
    return REL * abs(ref) + KAPPA * rss


def assert_dlambda(got: float, ref: float, rss: float) -> None:
    err = abs(got - ref)
    b = bound(ref, rss)
    assert err <= b, f"dlambda {got:.6g} vs oracle {ref:.6g}: error {err:.3g} > bound {b:.3g}"
    assert_rejects_plausible_bugs(ref, rss)


def assert_rejects_plausible_bugs(ref: float, rss: float) -> None:
    b = bound(ref, rss)
    if rss <= 1e-12 * (1.0 + abs(ref)):
        # Every per-row term vanishes (e.g. one visible key per row: y does
        # not depend on lambda); the bound is then ~0 and rejects any error.
        assert b <= 1e-9
        return
    assert b < 0.5 * rss, "the bound does not reject an error the size of one row's term"
    if abs(ref) > 0.05 * rss:
        # -dlambda (sign flip) is 2|dlambda| away, 0 (dropped term) |dlambda| away.
        assert b < 0.5 * abs(ref), "the bound does not reject a flipped or dropped lambda term"
