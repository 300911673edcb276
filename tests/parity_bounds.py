"""Bounds on how far a GPU decision can sit from the oracle's and still be
taken the other way, from the fp32 arithmetic each side does (derived
below, decision by decision). A GPU result that differs from the
oracle's is accepted only when the oracle reports the decision's margin below
its bound; everything else must match exactly.

u = 2^-24 is the fp32 rounding unit.

Top-k filter (dflash_rule.cuh): every weight, prefix sum and normaliser is
float-float, the weights' exp() within about 1e-9 (2^-29.9) relative, so a
kept probability is its exact value to 2^-29, rounded once to fp32
(relative error <= u + 2^-29 < 1.05 u).
- accept test u_i < p(d)/q(d): the GPU ratio is within 3.2u of the exact one,
  the oracle's within u, and u_i is exact: a decision can differ only when
  |u_i - p/q| <= 4.2u (p/q)                        -> ACCEPT_REL = 2^-21
- top-p cut RN(mass before) < top_p: the mass before is within 2^-29 on the
  GPU and exact on the oracle, each rounded to fp32; the test can differ
  only if top_p lies between the two roundings: |before - top_p| <= u +
  2^-29 <= 2^-22.9 top_p (top_p >= 1/2)             -> CUT_REL = 2^-21
- inverse CDF RN(u * total) < RN(cumulative weight), in probability units:
  the residual's weights max(0, p - q) come from fp32 p and q (error
  <= 1.05u (p + q) each, plus u max(0, p - q) for the subtraction), the sums
  are float-float, so each side is within 3.2u of the exact value, and the
  two fp32 roundings add at most 2u:               -> DRAW_ABS = 2^-21
Full-vocabulary filter: the draw is float-float over the whole row
(dflash_fullvocab.cu), no fp32 list values in between: each side within
2^-29 and two fp32 roundings (<= 2u)               -> FV_DRAW_ABS = 2^-22
Its accept test takes p(d) = exp((x_d - m)/T) / sum with a float-float
numerator and the row normaliser sum from the stream: each weight there is
2^a 2^c on the special-function unit (relative error below 2^-22.73 = 0.6u
each, measured over every fp32 argument in [-126, 0]; a = (logit - b) s for
b the maximum of the lane's block, c = (b - m) s once per block, then one
product rounding, u) of exponents rounded on the way: s = RN(log2(e) / T)
(1.22u), a product rounding (u) and, for fp32 logits, the difference (u)
in each part; a and c are <= 0, so their errors add to at most 3.22u of
|x|, x = (logit - m) s. A relative error e in the exponent x <= 0 changes
the weight by ln2 |x| e, and the weighted mean of |x| over the row is at
most its entropy in bits, <= log2 V = 17.92 at V = 248320:
<= 0.693 * 17.92 * 3.22u = 40u. Block sums are pairwise (<= 5u),
everything above them float-float. So
  sum:        <= 1.2u + u + 1.22u + 40u + 5u = 48.4u
  p(d), q(d): <= 48.4u + u (rounded once)           -> FV_PROB_REL = 2^-18
  the ratio (two of them, rounded) and the oracle's -> FV_ACCEPT_REL = 2^-17
Top-p over the full vocabulary (top-k off, top_p < 1; dflash_fvtp.cu): each
weight exp((x - m)/T) is float-float (2^-29.9 relative) and is rounded to
fixed point with f = 62 - ceil(log2 V) fractional bits (two roundings of half
a unit), so a sum of n <= V weights is exact up to n 2^-f <= V^2 2^-62
in units of the row's largest weight, 1, which every row's mass exceeds:
eps_V = V^2 2^-62 (2^-26 at V = 248320) as a fraction of the mass.
- the cut RN32(mass before / mass) < top_p: the GPU's fraction is within
  eps_V + 2^-29.9 of the exact one; the two decisions differ only when the
  two fp32 roundings straddle top_p, so the exact fraction is within
  eps_V + 2^-29.9 + u top_p of top_p        -> fvtp_cut_rel(V, top_p)
- p(d) = RN32(w(d) / kept mass): within u + eps_V + 2^-29.9 relative
  (1.31u at V = 248320)                       -> fvtp_prob_rel(V)
- the accept ratio: two such values and one fp32 division, the oracle's
  exact: 3.7u at V = 248320, under ACCEPT_REL = 8u
- the draw is the full-vocabulary one over the kept set: FV_DRAW_ABS.
"""
import math

U = 2.0 ** -24
ACCEPT_REL = 2.0 ** -21
CUT_REL = 2.0 ** -21
DRAW_ABS = 2.0 ** -21
FV_DRAW_ABS = 2.0 ** -22
FV_PROB_REL = 2.0 ** -18
FV_ACCEPT_REL = 2.0 ** -17

# the sampling-mode bar: rows (tokens and accept length) equal on >= 99.99%
ROW_BAR = 1e-4


def excused_topk(m_acc, m_cut, m_draw):
    """Whether a top-k request's oracle margins put one of its decisions
    within the GPU's rounding (then a different result is not an error)."""
    return m_acc < ACCEPT_REL or m_cut < CUT_REL or m_draw < DRAW_ABS


def excused_fullvocab(m_acc, m_draw):
    return m_acc < FV_ACCEPT_REL or m_draw < FV_DRAW_ABS


def fvtp_eps(V):
    """Bound on the fixed-point mass sums' error, as a fraction of the mass."""
    frac = 62 - math.ceil(math.log2(V)) if V > 1 else 62
    return V * 2.0 ** -frac + 2.0 ** -29.9


def fvtp_cut_rel(V, top_p):
    """The oracle's cut margin (relative to top_p) below which a top-p cut over
    the full vocabulary may be taken the other way."""
    return (fvtp_eps(V) + U * top_p) / top_p * 1.01


def fvtp_prob_rel(V):
    return (U + fvtp_eps(V)) * 1.01


def excused_fvtp(V, top_p, m_acc, m_cut, m_draw):
    return m_acc < ACCEPT_REL or m_cut < fvtp_cut_rel(V, top_p) or m_draw < FV_DRAW_ABS


def compare_rows(tok, ln, want_tok, want_len, excused, what=""):
    """Rows (tokens, accept length) must match the oracle unless excused(b);
    returns the number of differing rows."""
    import numpy as np

    same = np.all(tok == want_tok, axis=1) & (ln == want_len)
    bad = np.nonzero(~same)[0]
    for b in bad:
        assert excused(b), (f"{what} request {b}: gpu {tok[b].tolist()} len {ln[b]} vs oracle "
                            f"{want_tok[b].tolist()} len {want_len[b]}")
    return len(bad)
