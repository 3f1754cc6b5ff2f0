"""GPU parity of kvq_meter (finalisation, coverage counts, per-request ranking) against the oracle.

The meter states fed to the kernel are synthetic ln(A - 1) values (not decode
outputs), spanning the identity quantizer (-inf), the informative range, the
saturated range up to e^700, exact ties and non-finite cells.
"""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def kvq():
    import quantized_kv_cache_kvq_gb300 as m

    assert torch.cuda.is_available()
    m.load()
    return m


def test_meter_finalize_counts_and_ranking(kvq):
    from oracle import meter as OM

    L, B, H = 36, 5, 32
    rng = np.random.default_rng(9)
    la = rng.uniform(-12, 6, (L, B, H))
    la[0, 0, :4] = -np.inf
    la[1, 1, :3] = 700.0
    la[2, 2, 5:9] = -1.25          # exact ties
    la[3, 3, 0] = np.nan
    lb = rng.uniform(-15, 2, (L, B, H))
    la = la.astype(np.float32).astype(np.float64)
    lb = lb.astype(np.float32).astype(np.float64)
    state = np.zeros((L, B, H, 8), dtype=np.float32)
    state[..., 0] = la
    state[..., 1] = lb
    tau = 0.2
    p = kvq.meter_params(kvq.TIER_A | kvq.TIER_B, L, H, 256, 1e-3, tau)
    dev = "cuda"
    st = torch.from_numpy(state).to(dev)
    ma = torch.empty((L, B, H), device=dev)
    ra = torch.empty((L, B, H), device=dev)
    cb = torch.empty((L, B, H), device=dev)
    counts = torch.empty(4, dtype=torch.int32, device=dev)
    rank = torch.empty((B, L * H), dtype=torch.int32, device=dev)
    kvq.meter(st, L, B, H, p, ma, ra, counts, cert_b=cb, ranking=rank)
    torch.cuda.synchronize()
    m_ref, r_ref = OM.finalize(la)
    cb_ref, _ = OM.finalize(lb)
    got_m, got_r = ma.cpu().numpy(), ra.cpu().numpy()
    fin = np.isfinite(r_ref)
    assert np.allclose(got_m[fin], m_ref[fin], rtol=2e-6, atol=1e-7)
    assert np.allclose(got_r[fin], r_ref[fin], rtol=2e-6, atol=2e-6)
    assert np.all(np.isneginf(got_r[np.isneginf(r_ref)]))
    assert np.isnan(got_r[3, 3, 0])
    assert np.allclose(cb.cpu().numpy(), cb_ref, rtol=2e-6, atol=1e-7)
    c = counts.cpu().numpy()
    finite_m = np.where(np.isnan(la), np.nan, m_ref)
    assert c[0] == OM.coverage(finite_m, tau)
    assert c[1] == OM.coverage(cb_ref, tau)
    assert c[2] == 1 and c[3] == L * B * H
    # ranking per request over (layer, head), highest raw first, ties to the lower index.  The
    # kernel ranks its own binary32 raw scores; compare against the oracle's order of those scores
    # where the binary32 values are distinct from their neighbours in the oracle order.
    rk = rank.cpu().numpy()
    ref_rank = OM.rank_cells(got_r.transpose(1, 0, 2).astype(np.float64))
    assert np.array_equal(rk, ref_rank)
    # and the order agrees with the float64 raw scores up to binary32 ties
    for b in range(B):
        s64 = r_ref.transpose(1, 0, 2).reshape(B, -1)[b][rk[b]]
        s64 = np.where(np.isnan(s64), np.inf, s64)
        s64 = np.where(np.isneginf(s64), -1e300, s64)   # identity-quantizer cells: equal ranks
        assert np.all(np.diff(s64) <= 1e-5 * np.maximum(1, np.abs(s64[1:])))
