"""Exact vs compressed decode attention, total variation, and the two-tier meter (oracle; test infrastructure).

Everything is float64 and follows WitCert (arXiv 2607.28699):

* §3 "Setup and notation": p and p~ are the softmax attention distributions over
  the S cached tokens from exact and compressed keys; the metered quantity is
  TV(p, p~) = 1/2 sum_t |p_t - p~_t|, reported as min(1, .) because TV <= 1.
* §3 Theorem 1: with A = E_p~[e^{c}] and |eps_t| <= c_t, TV <= 1/2 (A^2 - 1).
  The page evaluates A in the log domain, returns 1 when it overflows and
  leaves c itself untouched: here the meter state is ln(A - 1), computed by
  log-sum-exp, so it never overflows and c is never clipped.
* §4.1 Theorem 2: c_t = (1/sqrt(d)) sum_b ||q_b|| w_{t,b} (the kernel form uses
  sm_scale in place of 1/sqrt(d)); w is the stored fp16 witness.
* §4.2: Tier B radius u_t = sqrt(2 varsigma_t^2 log(2S/delta_loc)) with
  varsigma_t^2 = (1/d) sum_c q_c^2 s_{c,t}^2 / 12, delta_loc = delta_req/(L*H*T);
  with one scale per (token, kv head) this is
  u_t = sm_scale * ||q|| * s_t * sqrt(2 ln(2S/delta_loc) / 12) (§6.2.2 hoists the sqrt).
  This library's dither lies on a 256-point grid (oracle.philox), so the rounding
  error of each element has a mean of at most 2^-9 LSB; the radius adds that
  deterministic part, sm_scale * s_t * ||q||_1 * 2^-9.  With one scale per group of
  G_c channels (§6.2.3), varsigma_t keeps the per-channel sum:
  u_t = sm_scale (kappa sqrt(sum_g ||q_g||^2 s_{g,t}^2) + 2^-9 sum_g ||q_g||_1 s_{g,t}).
* §4.3: meter = min(1, 1/2 (A^2 - 1)); the raw value (kept as a log score
  ln(1/2 (A^2 - 1))) is a risk score with no guarantee above 1.
* "Compress the shared cartridge", "One kernel spans cartridge and live KV":
  the shared prefix and the request's live suffix form one logical sequence
  under one softmax (the caller concatenates them before calling this module).

The output is o = sum_t p~_t v_hat_t with the dequantized values.

Value side (WitCert §3, the statement that TV propagates linearly to the output):
with y = sum_t p_t v_t the exact output and y_hat = sum_t p~_t v_hat_t,

    ||y - y_hat|| <= 2 TV max_t ||v_t|| + sum_t p~_t rho^v_t,   rho^v_t = ||v_hat_t - v_t||,

(split y - y_hat = sum_t (p_t - p~_t) v_t + sum_t p~_t (v_t - v_hat_t) and bound each sum by
the triangle inequality).  With the meter in place of TV and the stored fp16 round-up
value witness (rho^v_t, ||v_t||), the output-error bound is
2 min(1, 1/2 (A^2 - 1)) Vmax + R with R = sum_t p~_t rho^v_t and Vmax = max_t ||v_t||.

Alternative bound shapes (WitCert §4.3 Proposition 1 and the det-tanh shape of its comparison):
* two-sided: with A^- = E_p~[e^{-c}], TV <= 1/2 (A/A^- - A^-/A); neither this nor 1/2 (A^2 - 1) dominates,
  so the bound is the minimum of the two (and of 1);
* det-tanh: with every |eps_t| <= c_t, TV <= tanh(max_t c_t), a data-independent worst case merged by max.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from .philox import subtractive_error_bias_bound
from .quant import HEAD_DIM, N_BANDS

__all__ = [
    "DecodeResult",
    "logsumexp",
    "log_expm1",
    "softmax",
    "total_variation",
    "band_q_norms",
    "tier_a_radius",
    "tier_b_radius",
    "tier_b_radius_bypass",
    "tier_b_radius_groups",
    "log_a_minus_1",
    "meter_from_log_am1",
    "raw_log_score",
    "decode_head",
    "flawed_dispersion_bound",
    "two_sided_bound",
    "value_side",
    "output_error_bound",
    "one_minus_a_minus",
    "two_sided_meter",
    "det_tanh_bound",
]


def logsumexp(a: np.ndarray, axis=-1) -> np.ndarray:
    a = np.asarray(a, dtype=np.float64)
    m = np.max(a, axis=axis, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    with np.errstate(divide="ignore"):
        out = np.log(np.sum(np.exp(a - m), axis=axis, keepdims=True)) + m
    return np.squeeze(out, axis=axis)


def log_expm1(c: np.ndarray) -> np.ndarray:
    """ln(e^c - 1) for c >= 0, accurate for tiny and huge c (-inf at c = 0)."""
    c = np.asarray(c, dtype=np.float64)
    with np.errstate(divide="ignore"):
        small = np.log(np.expm1(np.minimum(c, 1.0)))
        large = c + np.log1p(-np.exp(-np.maximum(c, 1.0)))
    return np.where(c < 1.0, small, large)


def softmax(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return np.exp(x - logsumexp(x)[..., None])


def total_variation(p: np.ndarray, p_t: np.ndarray) -> np.ndarray:
    """TV(p, p~) = 1/2 sum_t |p_t - p~_t| (WitCert §3)."""
    return 0.5 * np.sum(np.abs(p - p_t), axis=-1)


def band_q_norms(q: np.ndarray) -> np.ndarray:
    """||q_b|| over the 16 half-split RoPE bands, q [..., 128] -> [..., 16]."""
    q = np.asarray(q, dtype=np.float64)
    half = HEAD_DIM // 2
    per = half // N_BANDS
    lo = q[..., :half].reshape(q.shape[:-1] + (N_BANDS, per))
    hi = q[..., half:].reshape(q.shape[:-1] + (N_BANDS, per))
    return np.sqrt(np.sum(lo * lo, -1) + np.sum(hi * hi, -1))


def tier_a_radius(q: np.ndarray, w: np.ndarray, sm_scale: float) -> np.ndarray:
    """c_t = sm_scale * sum_b ||q_b|| w_{t,b} (WitCert §4.1, Theorem 2).  q [128], w [S, 16] -> [S]."""
    return sm_scale * (np.asarray(w, dtype=np.float64) @ band_q_norms(q))


def tier_b_radius(q: np.ndarray, s_k: np.ndarray, sm_scale: float, seq_len: int,
                  delta_req: float, n_layers: int, n_q_heads: int, n_steps: int) -> np.ndarray:
    """Tier B radius of every token (WitCert §4.2), delta_loc = delta_req/(L H T):

        u_t = sm_scale s_t (||q|| sqrt(2 ln(2S/delta_loc)/12) + ||q||_1 beta),  beta = 2^-9.

    The first term is the page's sub-Gaussian radius (the hoisted square root of §6.2.2).  The
    second covers the dither grid: with xi uniform on 256 points instead of the continuum, each
    element's rounding error has a mean of at most beta in LSB units (its centred part keeps the
    variance proxy 1/12), so the error's mean contributes at most s_t ||q||_1 beta to eps_t.
    """
    delta_loc = delta_req / (n_layers * n_q_heads * n_steps)
    kappa = math.sqrt(2.0 * math.log(2.0 * seq_len / delta_loc) / 12.0)
    q = np.asarray(q, dtype=np.float64)
    qn = float(np.sqrt(np.sum(q ** 2)))
    q1 = float(np.sum(np.abs(q)))
    return sm_scale * (qn * kappa + q1 * subtractive_error_bias_bound()) * np.asarray(s_k, dtype=np.float64)


def tier_b_radius_groups(q: np.ndarray, s_kg: np.ndarray, sm_scale: float, seq_len: int,
                         delta_req: float, n_layers: int, n_q_heads: int, n_steps: int) -> np.ndarray:
    """Tier B radius with one key scale per token per channel group (WitCert §4.2 with the per-channel
    scales of §6.2.3): s_kg [S, n_groups], group g = channels [g G_c, (g + 1) G_c), G_c = 128 / n_groups.

        u_t = sm_scale (kappa sqrt(sum_c q_c^2 s_{g(c),t}^2) + 2^-9 sum_c |q_c| s_{g(c),t}),
        kappa = sqrt(2 ln(2S/delta_loc) / 12),

    the sub-Gaussian radius of sum_c q_c s_{g(c),t} (code_c - xi_c - x_c / s_{g(c),t}) (independent
    per-channel errors with variance proxy s^2 / 12) plus the dither grid's bias bound per channel.
    """
    delta_loc = delta_req / (n_layers * n_q_heads * n_steps)
    kappa = math.sqrt(2.0 * math.log(2.0 * seq_len / delta_loc) / 12.0)
    s = np.asarray(s_kg, dtype=np.float64)
    n_groups = s.shape[-1]
    qg = np.asarray(q, dtype=np.float64).reshape(n_groups, HEAD_DIM // n_groups)
    q2 = np.sum(qg * qg, axis=-1)          # ||q_g||^2
    q1 = np.sum(np.abs(qg), axis=-1)       # ||q_g||_1
    return sm_scale * (kappa * np.sqrt((s * s) @ q2) + subtractive_error_bias_bound() * (s @ q1))


FP16_REL = 2.0 ** -11   # |RN_fp16(x) - x| <= 2^-11 |RN_fp16(x)| for normal results ...
FP16_ABS = 2.0 ** -25   # ... and <= 2^-25 in the subnormal range


def tier_b_radius_bypass(q: np.ndarray, s_k: np.ndarray, k_hat_bypass: np.ndarray, channels, sm_scale: float,
                         seq_len: int, delta_req: float, n_layers: int, n_q_heads: int, n_steps: int) -> np.ndarray:
    """Tier B radius with the fixed-channel bypass (WitCert §6.2.5, §4.2).

    The dither (probabilistic) term uses the query restricted to the INT8 channels (the bypassed
    channels leave the variance term); the bypassed channels' fp16 rounding is deterministic and
    added by Cauchy-Schwarz: |q_O . r_O| <= ||q_O|| (2^-11 ||k_hat_O|| + sqrt(2m) 2^-25).
    ``k_hat_bypass`` [S, 2m]: the stored fp16 values of the bypassed channels.
    """
    q = np.asarray(q, dtype=np.float64)
    ch = np.asarray(channels)
    keep = np.ones(q.shape[-1], dtype=bool)
    keep[ch] = False
    u = tier_b_radius(q[keep], s_k, sm_scale, seq_len, delta_req, n_layers, n_q_heads, n_steps)
    qo = float(np.sqrt(np.sum(q[ch] ** 2)))
    ko = np.sqrt(np.sum(np.asarray(k_hat_bypass, dtype=np.float64) ** 2, axis=-1))
    return u + sm_scale * qo * (FP16_REL * ko + math.sqrt(len(ch)) * FP16_ABS)


def log_a_minus_1(log_p: np.ndarray, radius: np.ndarray) -> float:
    """ln(A - 1) with A - 1 = sum_t p~_t (e^{c_t} - 1), evaluated in the log domain (WitCert §3)."""
    terms = np.asarray(log_p, dtype=np.float64) + log_expm1(radius)
    if not np.any(np.isfinite(terms)):
        return -math.inf
    return float(logsumexp(terms))


def meter_from_log_am1(lam1) -> np.ndarray:
    """min(1, 1/2 (A^2 - 1)) from ln(A - 1) (WitCert §4.3); A - 1 >= e^0 = 1 always saturates."""
    lam1 = np.asarray(lam1, dtype=np.float64)
    with np.errstate(over="ignore"):
        am1 = np.exp(np.minimum(lam1, 1.0))
    return np.minimum(1.0, 0.5 * am1 * (am1 + 2.0))


def raw_log_score(lam1) -> np.ndarray:
    """ln(1/2 (A^2 - 1)) = ln(A-1) + ln(A+1) - ln 2, finite for any finite ln(A-1) (WitCert §4.3)."""
    lam1 = np.asarray(lam1, dtype=np.float64)
    with np.errstate(invalid="ignore"):   # NaN states (non-finite inputs) stay NaN
        return lam1 + np.logaddexp(math.log(2.0), lam1) - math.log(2.0)


@dataclass
class DecodeResult:
    out: np.ndarray          # [H, 128] compressed-attention output
    lse: np.ndarray          # [H] log-sum-exp of the compressed logits
    tv: np.ndarray           # [H] exact total variation between p and p~
    log_am1_a: np.ndarray    # [H] ln(A - 1), Tier A
    meter_a: np.ndarray      # [H] min(1, 1/2 (A^2 - 1)), Tier A
    raw_a: np.ndarray        # [H] ln(1/2 (A^2 - 1)), Tier A
    log_am1_b: np.ndarray    # [H] ln(A_B - 1), Tier B (nan when not requested)
    cert_b: np.ndarray       # [H] min(1, 1/2 (A_B^2 - 1)) (nan when not requested)
    c_max: np.ndarray        # [H] max_t c_t (diagnostic)
    value_r: np.ndarray | None = None      # [H] R = sum_t p~_t rho^v_t (value witness given)
    value_vmax: float | None = None        # max_t ||v_t|| (value witness given)
    out_bound_a: np.ndarray | None = None  # [H] 2 meter_a Vmax + R
    out_err: np.ndarray | None = None      # [H] ||y - y_hat|| with exact keys and values (v_exact given)
    one_minus_a_minus: np.ndarray | None = None  # [H] 1 - A^- = E_p~[1 - e^{-c}] (Tier A radius)
    meter_two_sided: np.ndarray | None = None    # [H] min(1, 1/2 (A^2 - 1), 1/2 (A/A^- - A^-/A))
    meter_tanh: np.ndarray | None = None         # [H] tanh(max_t c_t)


def decode_head(q: np.ndarray, k_exact: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray,
                w: np.ndarray, sm_scale: float, s_k: np.ndarray | None = None,
                tier_b: dict | None = None, vw: np.ndarray | None = None,
                v_exact: np.ndarray | None = None, bypass: dict | None = None) -> DecodeResult:
    """Decode attention of H query heads that share one kv head's cache.

    q [H, 128] (the query values exactly as the kernel reads them), k_exact
    [S, 128] (the binary32 post-RoPE keys), k_hat / v_hat [S, 128] (exact
    dequantized cache), w [S, 16] (witness values), s_k [S] (key scales, Tier B; [S, n_groups] for
    one scale per token per channel group, WitCert §6.2.3),
    tier_b = dict(delta_req, n_layers, n_q_heads, n_steps) or None, vw [S, 2] (value witness
    values: rho^v, ||v||) or None, v_exact [S, 128] (the binary32 values) or None, bypass =
    dict(channels [2m], values [S, 2m]) for keys stored with the fixed-channel outlier bypass (Tier B).
    """
    q = np.asarray(q, dtype=np.float64)
    H = q.shape[0]
    S = k_hat.shape[0]
    x_exact = sm_scale * (q @ np.asarray(k_exact, dtype=np.float64).T)   # [H, S]
    x_comp = sm_scale * (q @ np.asarray(k_hat, dtype=np.float64).T)
    lse = logsumexp(x_comp)
    log_pt = x_comp - lse[:, None]
    p_t = np.exp(log_pt)
    p = softmax(x_exact)
    out = p_t @ np.asarray(v_hat, dtype=np.float64)
    tv = total_variation(p, p_t)
    la = np.empty(H)
    lb = np.full(H, np.nan)
    cmax = np.empty(H)
    om = np.empty(H)
    for h in range(H):
        c = tier_a_radius(q[h], w, sm_scale)
        cmax[h] = float(np.max(c)) if S else 0.0
        la[h] = log_a_minus_1(log_pt[h], c)
        om[h] = one_minus_a_minus(p_t[h], c)
        if tier_b is not None:
            if bypass is not None:
                u = tier_b_radius_bypass(q[h], s_k, bypass["values"], bypass["channels"], sm_scale, S, **tier_b)
            elif np.ndim(s_k) == 2:
                u = tier_b_radius_groups(q[h], s_k, sm_scale, S, **tier_b)
            else:
                u = tier_b_radius(q[h], s_k, sm_scale, S, **tier_b)
            lb[h] = log_a_minus_1(log_pt[h], u)
    res = DecodeResult(out=out, lse=lse, tv=tv, log_am1_a=la, meter_a=meter_from_log_am1(la),
                       raw_a=raw_log_score(la), log_am1_b=lb,
                       cert_b=np.where(np.isnan(lb), np.nan, meter_from_log_am1(lb)), c_max=cmax)
    res.one_minus_a_minus = om
    res.meter_two_sided = two_sided_meter(la, om)
    res.meter_tanh = det_tanh_bound(cmax)
    if vw is not None:
        res.value_r, res.value_vmax = value_side(p_t, vw)
        res.out_bound_a = output_error_bound(res.meter_a, res.value_r, res.value_vmax)
    if v_exact is not None:
        y = p @ np.asarray(v_exact, dtype=np.float64)
        res.out_err = np.sqrt(np.sum((y - out) ** 2, axis=-1))
    return res


def value_side(p_t: np.ndarray, vw: np.ndarray):
    """R = sum_t p~_t rho^v_t per head (p_t [H, S]) and Vmax = max_t ||v_t|| from value witness values
    vw [S, 2] = (rho^v_t, ||v_t||).  Vmax is 0 for an empty sequence."""
    vw = np.asarray(vw, dtype=np.float64)
    r = np.asarray(p_t, dtype=np.float64) @ vw[:, 0]
    vmax = float(np.max(vw[:, 1])) if vw.shape[0] else 0.0
    return r, vmax


def output_error_bound(tv_bound, r, vmax):
    """WitCert §3: ||y - y_hat|| <= 2 TV max_t ||v_t|| + sum_t p~_t rho^v_t, with a TV bound for TV."""
    return 2.0 * np.asarray(tv_bound, dtype=np.float64) * vmax + np.asarray(r, dtype=np.float64)


def flawed_dispersion_bound(p_t: np.ndarray, c: np.ndarray) -> float:
    """WitCert §3 eq. (1), the plausible but unsound certificate (kept as a regression guard).

    1/2 e^{2 c_max} ( E_p~|c - c_bar| + c_bar (e^{c_max} - 1) ), c_bar = E_p~[c].
    """
    p_t = np.asarray(p_t, dtype=np.float64)
    c = np.asarray(c, dtype=np.float64)
    cbar = float(p_t @ c)
    cmax = float(np.max(c))
    return 0.5 * math.exp(2 * cmax) * (float(p_t @ np.abs(c - cbar)) + cbar * (math.exp(cmax) - 1.0))


def two_sided_bound(a: float, a_minus: float) -> float:
    """WitCert §4.3 Proposition 1: TV <= 1/2 (A/A^- - A^-/A) with A^- = E_p~[e^{-c}]."""
    return 0.5 * (a / a_minus - a_minus / a)


def one_minus_a_minus(p_t: np.ndarray, c: np.ndarray) -> float:
    """1 - A^- = E_p~[1 - e^{-c}] (WitCert §4.3 Proposition 1), computed without cancellation."""
    c = np.asarray(c, dtype=np.float64)
    return float(np.asarray(p_t, dtype=np.float64) @ (-np.expm1(-c))) if c.size else 0.0


def two_sided_meter(lam1, om) -> np.ndarray:
    """min(1, 1/2 (A^2 - 1), 1/2 (A/A^- - A^-/A)) from ln(A - 1) and 1 - A^- (Proposition 1 and Theorem 1)."""
    lam1 = np.asarray(lam1, dtype=np.float64)
    om = np.asarray(om, dtype=np.float64)
    one_sided = meter_from_log_am1(lam1)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        a = 1.0 + np.exp(lam1)
        am = 1.0 - om
        ts = 0.5 * (a / am - am / a)
    ts = np.where(np.isfinite(ts), ts, 1.0)
    return np.minimum(one_sided, np.minimum(1.0, ts))


def det_tanh_bound(c_max) -> np.ndarray:
    """tanh(max_t c_t): the data-independent worst-case shape TV <= tanh(max |eps|)."""
    return np.tanh(np.asarray(c_max, dtype=np.float64))
