"""Meter finalisation, coverage at tau, and per-request risk ranking (oracle; test infrastructure).

WitCert §4.3: the sound meter is min(1, 1/2 (A^2 - 1)); the raw value above
saturation carries no guarantee but ranks risk; certified gating uses tau < 1,
risk-ranked gating tau >= 1.  WitCert §6.2.4 ("Certificate telemetry in
production"): certificates are aggregated on the device; coverage is the share
of (layer, head) cells under tau; non-finite values are counted separately.

Ranking reading (the pages do not fix an order for ties): within one request,
(layer, q-head) cells are ordered by raw log score, highest first; equal scores
keep the lower flat index l * H + h first.
"""
from __future__ import annotations

import numpy as np

from .attention import meter_from_log_am1, raw_log_score

__all__ = ["finalize", "coverage", "rank_cells"]


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
