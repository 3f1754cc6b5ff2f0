"""Meter finalisation, coverage at tau, and per-request risk ranking (oracle; test infrastructure).

WitCert §4.3: the sound meter is min(1, 1/2 (A^2 - 1)); the raw value above
saturation carries no guarantee but ranks risk; certified gating uses tau < 1,
risk-ranked gating tau >= 1.  WitCert §6.2.4 ("Certificate telemetry in
production"): certificates are aggregated on the device; coverage is the share
of (layer, head) cells under tau; non-finite values are counted separately.

Gate support (WitCert §6.3.5 "Block-level paging"): A = sum_t p~_t e^{c_t} decomposes over blocks,
and replacing block j by its exact values lowers A - 1 by its contribution
sum_{t in j} p~_t (e^{c_t} - 1) (the compressed distribution held fixed); blocks are paged in in
decreasing order of contribution until the meter min(1, 1/2 (A^2 - 1)) is at or below tau.  Here a
block is one 16-token page; larger blocks are sums of pages.

Ranking reading (the pages do not fix an order for ties): within one request,
(layer, q-head) cells are ordered by raw log score, highest first; equal scores
keep the lower flat index l * H + h first.
"""
from __future__ import annotations

import numpy as np

from .attention import meter_from_log_am1, raw_log_score

__all__ = ["finalize", "coverage", "rank_cells", "page_log_contrib", "greedy_page_in"]


def finalize(log_am1: np.ndarray):
    """(meter, raw) from ln(A - 1) values of any shape."""
    return meter_from_log_am1(log_am1), raw_log_score(log_am1)


def coverage(meter: np.ndarray, tau: float) -> int:
    """Number of cells whose meter is finite and strictly below tau."""
    m = np.asarray(meter, dtype=np.float64)
    return int(np.sum(np.isfinite(m) & (m < tau)))


def rank_cells(raw: np.ndarray) -> np.ndarray:
    """raw [B, L, H] -> [B, L*H] flat cell indices, highest raw first, ties to the lower index.

    NaN scores (non-finite inputs) rank first, as the most urgent.
    """
    raw = np.asarray(raw, dtype=np.float64)
    B = raw.shape[0]
    flat = raw.reshape(B, -1)
    key = np.where(np.isnan(flat), np.inf, flat)
    idx = np.arange(flat.shape[1])
    out = np.empty(flat.shape, dtype=np.int64)
    for b in range(B):
        # lexsort: last key is primary -> sort by -key, then by index
        out[b] = np.lexsort((idx, -key[b]))
    return out


def page_log_contrib(x: np.ndarray, c: np.ndarray, page: int = 16) -> np.ndarray:
    """ln sum_{t in page} e^{x_t} (e^{c_t} - 1) per page (natural log, not normalised) for logits x [S] and
    radii c [S]; -inf for a page whose tokens all have c = 0.  exp(result - lse(x)) is the page's
    contribution to A - 1."""
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(c, dtype=np.float64)
    n = (len(x) + page - 1) // page
    out = np.full(n, -np.inf)
    with np.errstate(divide="ignore"):
        term = x + np.log(np.expm1(c))  # ln(e^x (e^c - 1)); -inf where c = 0
    for j in range(n):
        t = term[j * page:(j + 1) * page]
        m = np.max(t) if t.size else -np.inf
        if np.isfinite(m):
            out[j] = m + np.log(np.sum(np.exp(t - m)))
    return out


def greedy_page_in(contrib: np.ndarray, a_minus_1: float, tau: float, max_pages: int | None = None):
    """Pages to page in (indices, highest contribution first, ties to the lower index) so that
    1/2 (A'^2 - 1) <= tau with A' - 1 = (A - 1) - sum of the chosen contributions; the shortest such
    prefix of the order.  ``max_pages`` caps the returned list (the count is not capped)."""
    contrib = np.asarray(contrib, dtype=np.float64)
    target = np.sqrt(1.0 + 2.0 * tau) - 1.0   # largest A - 1 with 1/2 (A^2 - 1) <= tau
    order = np.lexsort((np.arange(contrib.size), -contrib))
    rest, k = float(a_minus_1), 0
    while rest > target and k < contrib.size:
        rest -= contrib[order[k]]
        k += 1
    chosen = order[:k]
    return k, (chosen if max_pages is None else chosen[:max_pages])
