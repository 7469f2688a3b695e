"""Pins for the oracle's layout, capacity bound and expand-scatter.

The layout is checked by brute force on tiny inputs against a construction
by sorting (a different algorithm from the oracle's counting sort), and by
the invariants the method implies on the seeded workloads: every valid pair
appears exactly once, psum is the inclusive prefix with only earlier
experts aligned, segment starts and the total are multiples of the
alignment, labels are non-decreasing and -1 only past the aligned total.
"""
import itertools

import numpy as np
import pytest

import synth


def _by_sorting(ids, E, align, n_valid, M_cap, block_m=128):
    """Rows by sorting the valid pairs on (expert, token, k) and laying the
    experts out one after another, each padded up to the alignment."""
    T, K = ids.shape
    pairs = sorted((int(ids[t, k]), t, k) for t in range(n_valid) for k in range(K)
                   if 0 <= ids[t, k] < E)
    src2dst = -np.ones((T, K), np.int64)
    m_idx = -np.ones(M_cap, np.int64)
    start, psum, tiles = [], [], [0]
    row = 0
    for e in range(E):
        mine = [p for p in pairs if p[0] == e]
        start.append(row)
        for j, (_, t, k) in enumerate(mine):
            src2dst[t, k] = row + j
        psum.append(row + len(mine))
        seg = -(-len(mine) // align) * align
        m_idx[row:row + seg] = e
        tiles.append(tiles[-1] + -(-seg // block_m))
        row += seg
    return dict(start=start, psum=psum, total=row, src2dst=src2dst, m_indices=m_idx,
                tile_prefix=tiles)


def test_layout_brute_force_tiny(orc):
    n_cases = 0
    for T, K, E in [(1, 1, 1), (2, 2, 2), (3, 2, 3), (3, 1, 3), (2, 2, 3)]:
        vals = range(-1, E)
        for flat in itertools.product(vals, repeat=T * K):
            ids = np.array(flat, np.int32).reshape(T, K)
            for align in (1, 2, 3, 4):
                for n_valid in range(T + 1):
                    M_cap = T * K * align + 2
                    got = orc.layout(ids, E, align, n_valid, M_cap, block_m=2)
                    ref = _by_sorting(ids, E, align, n_valid, M_cap, block_m=2)
                    assert got["rc"] == 0
                    assert list(got["start"]) == ref["start"]
                    assert list(got["psum"]) == ref["psum"]
                    assert got["total"] == ref["total"]
                    assert np.array_equal(got["src2dst"], ref["src2dst"])
                    assert np.array_equal(got["m_indices"], ref["m_indices"])
                    assert list(got["tile_prefix"]) == ref["tile_prefix"]
                    n_cases += 1
    assert n_cases > 10000


def test_psum_matches_the_review_definition(orc):
    # psum[i] = align(psum[i-1]) + count_i (inclusive, only earlier experts
    # aligned); worked by hand for counts (3, 0, 6, 1), align 4:
    # psum = 3, align(3)+0 = 4, align(4)+6 = 10, align(10)+1 = 13.
    ids = np.array([[0, 2], [0, 2], [0, 2], [2, 3], [2, 2]], np.int32)
    lay = orc.layout(ids, 4, 4, 5, 64)
    assert list(lay["psum"]) == [3, 4, 10, 13]
    assert list(lay["start"]) == [0, 4, 4, 12]
    assert lay["total"] == 16


def _invariants(lay, ids, E, align, n_valid, M_cap):
    T, K = ids.shape
    s2d, m_idx, start, psum = lay["src2dst"], lay["m_indices"], lay["start"], lay["psum"]
    total = lay["total"]
    valid = np.zeros((T, K), bool)
    valid[:n_valid] = (ids[:n_valid] >= 0) & (ids[:n_valid] < E)
    # every valid pair exactly once, into [0, total), on a row of its expert
    assert (s2d[valid] >= 0).all() and (s2d[~valid] == -1).all()
    rows = s2d[valid]
    assert len(np.unique(rows)) == rows.size and (rows < total).all()
    assert (m_idx[rows] == ids[valid]).all()
    counts = np.bincount(ids[valid], minlength=E)
    assert (np.diff(np.concatenate([[0], psum])) >= 0).all()
    assert (np.asarray(start) % align == 0).all() and total % align == 0
    assert total == int(sum(-(-c // align) * align for c in counts))
    assert (np.asarray(psum) - np.asarray(start) == counts).all()
    assert (np.diff(m_idx[:total]) >= 0).all() and (m_idx[:total] >= 0).all()
    assert (m_idx[total:M_cap] == -1).all()
    assert total <= M_cap
    # within an expert, rows follow ascending (t, k)
    for e in range(E):
        tk = np.argwhere(valid & (ids == e))
        r = s2d[tk[:, 0], tk[:, 1]]
        assert (np.diff(r) == 1).all() and (r.size == 0 or r[0] == start[e])


@pytest.mark.parametrize("cfg", synth.PARITY_CONFIGS + tuple(synth.config_by_name(n) for n in ("uniform_t4096_h4096", "zipf_t16384_h7168", "padded_t32768_valid6000_h4096")),
                         ids=lambda c: c.name)
def test_layout_invariants_on_workloads(orc, cfg):
    d = synth.generate(cfg, with_weights=False)
    ids = d["topk_ids"].numpy()
    M_cap = orc.expanded_capacity(cfg.T * cfg.K, cfg.E, cfg.align)
    lay = orc.layout(ids, cfg.E, cfg.align, cfg.valid_rows, M_cap)
    assert lay["rc"] == 0
    _invariants(lay, ids, cfg.E, cfg.align, cfg.valid_rows, M_cap)
    if cfg.routing == "zipf":
        counts = np.diff(np.concatenate([[0], lay["psum"]])) - np.diff(np.concatenate([[0], lay["start"]]))
        assert (np.asarray(lay["psum"]) == np.asarray(lay["start"])).sum() >= 1, "some expert empty"


def test_layout_bad_id_and_capacity_errors(orc):
    ids = np.array([[0, 5], [1, 1]], np.int32)
    lay = orc.layout(ids, 4, 2, 2, 16)
    assert lay["rc"] == -3 and lay["src2dst"][0, 1] == -1
    ids = np.array([[0, 1], [2, 3]], np.int32)
    assert orc.layout(ids, 4, 8, 2, 31)["rc"] == -2
    # rows past n_valid are never read: garbage ids there are no error
    ids = np.array([[0, 1], [99, -5]], np.int32)
    assert orc.layout(ids, 4, 2, 1, 16)["rc"] == 0


def test_capacity_is_the_max_over_all_routings(orc):
    for A in range(0, 9):
        for E in range(1, 5):
            for a in range(1, 5):
                best = 0
                for counts in itertools.product(range(A + 1), repeat=E):
                    if sum(counts) == A:
                        best = max(best, sum(-(-c // a) * a for c in counts))
                assert orc.expanded_capacity(A, E, a) == best, (A, E, a)


@pytest.mark.parametrize("cfg", synth.PARITY_CONFIGS, ids=lambda c: c.name)
def test_scatter_rows_are_their_tokens_and_gaps_are_zero(orc, cfg):
    d = orc.to_numpy_inputs(synth.generate(cfg, with_weights=False))
    M_cap = orc.expanded_capacity(cfg.T * cfg.K, cfg.E, cfg.align)
    lay = orc.layout(d["topk_ids"], cfg.E, cfg.align, d["n_valid"], M_cap)
    xe, xe_s, row_w = orc.scatter(d["x_q"], d["x_s"], d["scale_layout"], d["topk_w"], lay,
                                  d["n_valid"], cfg.E, cfg.align, M_cap)
    s2d = lay["src2dst"]
    written = np.zeros(M_cap, bool)
    for t in range(d["n_valid"]):
        for k in range(cfg.K):
            r = s2d[t, k]
            if r < 0:
                continue
            written[r] = True
            assert np.array_equal(xe[r], d["x_q"][t])
            assert row_w[r] == d["topk_w"][t, k]
            if d["scale_layout"] == orc.SCALE_F32:
                assert np.array_equal(xe_s[r].view(np.uint32), d["x_s"][t].view(np.uint32))
            else:
                assert np.array_equal(xe_s[:, r], d["x_s"][:, t])
    gaps = ~written
    assert (xe[gaps] == 0).all() and (row_w[gaps] == 0).all()
    if d["scale_layout"] == orc.SCALE_F32:
        assert (xe_s[gaps] == 0).all()
    else:
        assert (xe_s[:, gaps] == 0).all()
    # the gaps inside the aligned total are exactly the alignment padding
    pad = sum(-(-c // cfg.align) * cfg.align - c for c in
              np.asarray(lay["psum"]) - np.asarray(lay["start"]))
    assert gaps[:lay["total"]].sum() == pad
