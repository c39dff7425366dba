"""The parity checker's own rules, on the CPU: a GPU cache image stands in as an oracle image with
planted code changes, so the rules are shown to accept what is correct and reject what is not."""
import numpy as np
import pytest

from oracle import cache
from tests import harness as H
import synthetic as syn


def _identity_image():
    wl = syn.Workload("ties", syn.Shape(8, 2, 64, 16, 32, 2, 16, 1), [0], seed=5)
    s = wl.shape
    eye = np.eye(s.head_dim, dtype=np.float32)
    n = 400
    geom = H.geometry(s, syn.pages_for(n, s.page_size) + 1, 1)
    img = cache.CacheImage(geom)
    k, v = syn.kv_tokens(wl, 0, n)
    bt = np.arange(geom.num_pages, dtype=np.int32)[None, :]
    diag = cache.write_kv(img, 0, k, v, np.array([0, n], np.int32), np.zeros(1, np.int32), eye, eye,
                          4.0, 4.0, bt, np.zeros(1, np.int32))
    return img, diag


def _replant(img, diag, codes_k):
    kq = dict(diag["k"], codes=codes_k)
    out = cache.CacheImage(img.g)
    out.pool = img.pool.copy()
    out.store_history(0, diag["pages"], diag["slots"], kq, diag["v"])
    return out.pool


def test_exact_tie_takes_either_neighbour_but_nothing_else():
    img, diag = _identity_image()
    qd = diag["k"]
    ties = H._exact_ties(qd["y"], qd["scale"], qd["zero"], img.g.group_size)
    assert ties.any(), "BF16 inputs under R = I must produce exact ties"
    idx = tuple(np.argwhere(ties)[0])
    y = qd["y"][idx]
    g = idx[-1] // img.g.group_size
    t = (y - qd["zero"][idx[:-1] + (g,)]) / qd["scale"][idx[:-1] + (g,)]
    lo, hi = int(np.floor(t)), int(np.ceil(t))
    assert hi == lo + 1 and t == lo + 0.5
    other = hi if qd["codes"][idx] == lo else lo
    codes = qd["codes"].copy()
    codes[idx] = other
    pool = _replant(img, diag, codes)
    res = H.compare_history(pool, img.g, 0, diag, exact_ties=True)
    assert res["exempt"] == 0
    # without the tie rule the same change is a near-boundary exemption
    assert H.compare_history(pool, img.g, 0, diag)["exempt"] == 1
    # a code two steps away from a tie is wrong under either rule
    far = lo - 1 if lo >= 1 else hi + 1
    codes[idx] = far
    pool = _replant(img, diag, codes)
    with pytest.raises(AssertionError):
        H.compare_history(pool, img.g, 0, diag, exact_ties=True)


def test_code_change_away_from_a_boundary_is_rejected():
    img, diag = _identity_image()
    qd = diag["k"]
    near = H._near_code_boundary(qd["y"], qd["scale"], qd["zero"], img.g.group_size)
    idx = tuple(np.argwhere(~near)[0])
    codes = qd["codes"].copy()
    codes[idx] = (codes[idx] + 1) % 4
    pool = _replant(img, diag, codes)
    with pytest.raises(AssertionError, match="away from a rounding boundary"):
        H.compare_history(pool, img.g, 0, diag, exact_ties=True)


def _clipped_group_case(offset):
    """One token, one head, d = 64: group 0 holds 31 values at a clip threshold c = 12.3144 and one value
    c - 3 (m - offset), where m = 0.0443115234375 is the midpoint between the BF16 numbers 0.044189453125
    and 0.04443359375; so (max - min)/3 lies `offset` below a BF16 rounding boundary.  Returns the oracle
    diagnostics and a planted image whose group-0 scale is the neighbouring BF16 number (codes
    re-quantised with it), as a rotation that is not exact could produce."""
    from oracle import quant
    geom = cache.Geometry(1, 1, 64, 16, 32, 0, 1, 1, 1)
    c, m = 12.314421653747559, 0.0443115234375
    y = np.zeros((1, 1, 64))
    y[0, 0, :32] = c
    y[0, 0, 27] = c - 3.0 * (m - offset)
    y[0, 0, 32:] = np.linspace(-1.0, 1.0, 32)
    codes, scale, zero, mn, rng3 = quant.quantize_groups(y, 32)
    assert scale[0, 0, 0] == 0.044189453125
    qd = {"y": y, "codes": codes, "scale": scale, "zero": zero, "mn": mn, "rng3": rng3}
    diag = {"b": np.zeros(1, np.int64), "t": np.zeros(1, np.int64), "k": qd, "v": qd,
            "pages": np.zeros(1, np.int64), "slots": np.zeros(1, np.int64)}
    s2 = scale.copy()
    s2[0, 0, 0] = 0.04443359375
    planted = cache.CacheImage(geom)
    planted.store_history(0, diag["pages"], diag["slots"], dict(qd, scale=s2, codes=quant.quantize_with(y, s2, zero, 32)),
                          qd)
    return planted.pool, geom, diag


def test_scale_of_a_narrow_group_of_large_values_is_judged_on_their_magnitude():
    # 2e-7 below the boundary: outside 1e-6 of the range (4.4e-8) but inside 1e-6 of the values (1.2e-5)
    pool, geom, diag = _clipped_group_case(2e-7)
    res = H.compare_history(pool, geom, 0, diag, enforce_budget=False)
    kinds = [e[0] for e in res["list"]]
    assert kinds.count("K-scale") == 1 and "K-zero" not in kinds
    # 5e-5 below the boundary is outside either window: a wrong scale
    pool, geom, diag = _clipped_group_case(5e-5)
    with pytest.raises(AssertionError, match="scale/zero differ outside the boundary rule"):
        H.compare_history(pool, geom, 0, diag, enforce_budget=False)


def test_exemption_budget_has_no_slack():
    res = {"elements": 10000, "exempt": 1, "list": []}
    H.check_budget(res)
    with pytest.raises(AssertionError, match="too many exemptions"):
        H.check_budget(dict(res, exempt=2))
