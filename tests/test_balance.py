"""CP load-balance report (document_masked_gqa_gb300.balance) against the
oracle's per-position pair counts, a hand-worked example, and properties:
the pages' chunk pairing balances a single document exactly, and the
document-aware alternative never balances worse."""
import numpy as np
import pytest

from document_masked_gqa_gb300 import balance
from document_masked_gqa_gb300 import workloads as wl
from oracle import cp as ocp
from oracle import flops as ofl

NAMES = ["tiny", "8b", "70b", "sparse", "405b-logu", "405b-1doc"]


def _explicit_rank_pairs(cu, batch, seq_len, cp_size, bounds):
    """Oracle-side count for arbitrary chunk bounds: sum over the rank's query
    positions of (position - start of its document + 1)."""
    start = ocp.doc_start(cu, batch, seq_len)
    n = 2 * cp_size
    out = np.zeros((cp_size, batch), dtype=np.int64)
    for b in range(batch):
        e = bounds[b]
        for r in range(cp_size):
            pos = np.r_[e[r]:e[r + 1], e[n - 1 - r]:e[n - r]]
            out[r, b] = int((pos - start[b, pos] + 1).sum())
    return out


@pytest.mark.parametrize("name", NAMES)
def test_rank_work_matches_oracle(name):
    w = wl.WORKLOADS[name]
    cu = wl.cu_doc_lens(w)
    got = balance.rank_work(cu, w.batch, w.seq_len, w.cp_size)
    for r in range(w.cp_size):
        want = ofl.pairs_per_head(cu, w.batch, w.seq_len, w.cp_size, r)
        assert np.array_equal(got[r], want), (name, r)
    # the ranks together hold every query once
    whole = ofl.pairs_per_head(cu, w.batch, w.seq_len, 1, 0)
    assert np.array_equal(got.sum(axis=0), whole)


def test_worked_example():
    # S = 16, CP = 2 (chunks of 4), documents [0, 6) and [6, 16).  A query at
    # p sees p - start + 1 keys: 1..6 in the first document, 1..10 in the
    # second.  Chunks: [0,4) 1+2+3+4 = 10; [4,8) 5+6+1+2 = 14;
    # [8,12) 3+4+5+6 = 18; [12,16) 7+8+9+10 = 34.  Rank 0 holds chunks 0 and
    # 3 (44), rank 1 chunks 1 and 2 (32).
    cu = np.array([0, 6, 16], dtype=np.int32)
    got = balance.rank_work(cu, 1, 16, 2)
    assert got[:, 0].tolist() == [44, 32]
    imb = balance.imbalance(got)
    assert imb["max_over_mean"] == pytest.approx(44 / 38)
    assert imb["slowest_over_fastest"] == pytest.approx(44 / 32)


@pytest.mark.parametrize("cp_size", [1, 2, 4, 16])
def test_single_document_is_balanced(cp_size):
    seq_len = 4096
    cu = np.array([0, seq_len], dtype=np.int32)
    got = balance.rank_work(cu, 1, seq_len, cp_size)
    assert len(set(got[:, 0].tolist())) == 1
    assert got[0, 0] == ofl.single_doc_pairs_closed_form(seq_len // (2 * cp_size), cp_size)
    assert balance.imbalance(got)["max_over_mean"] == 1.0


@pytest.mark.parametrize("name", NAMES)
def test_explicit_bounds_match_oracle(name):
    w = wl.WORKLOADS[name]
    cu = wl.cu_doc_lens(w)
    rng = np.random.default_rng(7)
    n = 2 * w.cp_size
    bounds = np.zeros((w.batch, n + 1), dtype=np.int64)
    for b in range(w.batch):
        inner = np.sort(rng.choice(np.arange(1, w.seq_len), size=n - 1, replace=False))
        bounds[b] = np.r_[0, inner, w.seq_len]
    got = balance.rank_work(cu, w.batch, w.seq_len, w.cp_size, bounds)
    assert np.array_equal(got, _explicit_rank_pairs(cu, w.batch, w.seq_len, w.cp_size, bounds))


@pytest.mark.parametrize("name,cp_size", [(n, None) for n in NAMES] + [("8b", 4), ("8b", 8),
                                                                     ("405b-logu", 4)])
def test_doc_aware_alternative(name, cp_size):
    w = wl.WORKLOADS[name]
    cp = cp_size or w.cp_size
    cu = wl.cu_doc_lens(w)
    rep = balance.report(cu, w.batch, w.seq_len, cp)
    bounds = np.asarray(rep["doc_aware"]["bounds"])
    n = 2 * cp
    assert bounds.shape == (w.batch, n + 1)
    assert (bounds[:, 0] == 0).all() and (bounds[:, -1] == w.seq_len).all()
    assert (np.diff(bounds, axis=1) > 0).all()
    assert rep["doc_aware"]["imbalance"]["max_over_mean"] <= rep["imbalance"]["max_over_mean"]
    # the alternative's work is counted the same way as the oracle counts it
    alt = np.asarray(rep["doc_aware"]["pairs_per_rank"])
    want = _explicit_rank_pairs(cu, w.batch, w.seq_len, cp, bounds).sum(axis=1)
    assert np.array_equal(alt, want)
    # and it moves no work between ranks that is not there
    assert alt.sum() == sum(rep["pairs_per_rank"])


def test_equal_work_bounds_on_the_grid():
    w = wl.WORKLOADS["405b-logu"]
    cu = wl.cu_doc_lens(w)
    b = balance.balanced_bounds(cu, w.batch, w.seq_len, 4, granule=256)
    assert (b % 256 == 0).all() and (np.diff(b, axis=1) > 0).all()
    chunks = [balance._segment_work(balance._docs_of_sample(cu, 0, w.seq_len), b[0, c], b[0, c + 1])
              for c in range(8)]
    # every chunk within a few granules' work of the ideal share
    assert max(chunks) / (sum(chunks) / 8) < 1.1


@pytest.mark.parametrize("name", ["tiny", "8b", "70b", "sparse", "405b-logu"])
def test_tile_counts_match_oracle_block_mask(name):
    """Host counts of full / partial tile pairs against the oracle's tile
    classes, which look at every element of the explicit mask."""
    from oracle import blockmask as ob
    w = wl.WORKLOADS[name]
    cu = wl.cu_doc_lens(w)
    ranks = w.ranks if name != "405b-logu" else (15,)  # the oracle's brute force is slow at 128K
    for r in ranks:
        got = balance.tile_counts(cu, w.batch, w.seq_len, w.cp_size, r, w.group)
        cls = ob.tile_classes(cu, w.batch, w.seq_len, w.cp_size, r, w.group)
        assert got["full"] == int((cls == ob.FULL).sum()), (name, r)
        assert got["partial"] == int((cls == ob.PARTIAL).sum()), (name, r)


def test_cost_fit_recovers_known_constants():
    """fit_costs on times made from known constants (plus tiny noise) returns
    them; predict_ms reproduces the times."""
    rng = np.random.default_rng(3)
    coef = np.array([2.0e-4, 5.0e-5, 1.0e-3, 0.03])
    feats = []
    for name in ["8b", "70b", "sparse", "405b-logu", "405b-1doc"]:
        w = wl.WORKLOADS[name]
        cu = wl.cu_doc_lens(w)
        for r in w.ranks:
            feats.append(balance.rank_costs(cu, w.batch, w.seq_len, w.cp_size, r, w.n_heads,
                                            w.n_kv_heads))
    feats = np.array(feats)
    times = balance.predict_ms(feats, coef) * (1 + 1e-6 * rng.standard_normal(len(feats)))
    got = balance.fit_costs(feats, times)
    assert np.allclose(got, coef, rtol=1e-3, atol=1e-6)
    assert np.allclose(balance.predict_ms(feats, got), times, rtol=1e-4)


def _slices_cover(work, counts):
    got = {}
    for unit, first, n, seg, split, slot in work["slices"]:
        got.setdefault(unit, []).append((first, n, seg))
    assert sorted(got) == list(range(len(counts)))
    for unit, parts in got.items():
        parts.sort()
        assert [p[2] for p in parts] == list(range(len(parts)))
        pos = 0
        for first, n, _ in parts:
            assert first == pos
            pos += n
        assert pos == counts[unit]


def test_kv_work_list_hand_case():
    """One list of 100 query tiles and three of 1 over 4 SMs: the mean is
    25.75 tiles per SM and the long list alone bounds the greedy makespan at
    100 (> 1.15 x 25.75), while from the second unit on every bound is at most
    26.5 (< 1.10 x 25.75): L = max(16, 1) = 16, so 7 segments (6 pool slots)
    of 15 or 14 tiles, ahead of the three short lists."""
    assert balance.SEG_MIN == 16
    counts = [1, 100, 1, 1]
    work = balance.kv_work_list(counts, 1, 4, 20)
    assert work["L"] == 16
    assert work["splits"] == [(1, 0, 7)]
    lens = [n for u, f, n, sg, sp, sl in work["slices"] if u == 1]
    assert lens == [15] * 2 + [14] * 5  # 100 = 7 x 14 + 2: the first 2 take one more
    assert [s[0] for s in work["slices"]] == [1] * 7 + [0, 2, 3]
    assert [s[5] for s in work["slices"][:7]] == [-1] + list(range(6))
    _slices_cover(work, counts)
    # a pool of 5 slots: L grows 16, 18 until ceil(100 / L) - 1 <= 5
    work = balance.kv_work_list(counts, 1, 4, 5)
    assert work["L"] == 18 and work["splits"] == [(1, 0, 6)]
    # no pool: no cut, the longest-first order
    work = balance.kv_work_list(counts, 1, 4, 0)
    assert work["L"] is None and work["splits"] == []
    assert [s[0] for s in work["slices"]] == [1, 0, 2, 3]


def test_kv_work_list_leaves_even_lists_alone():
    """1000 lists of 10 tiles on 152 SMs: the bound (75.7) is over 1.15 x the
    mean (65.8), but no length below 10 brings every bound within 1.10 x the
    mean before the last unit, so L = 10 = the longest list: nothing to cut."""
    work = balance.kv_work_list([10] * 1000, 1, 152, 1000)
    assert work["L"] is None
    assert [s[0] for s in work["slices"]] == list(range(1000))


@pytest.mark.parametrize("seed", range(6))
def test_kv_work_list_covers_every_list(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 300))
    counts = (rng.pareto(1.2, n) * 20).astype(int).tolist()
    for hkv, sms, cap in [(1, 152, 512), (8, 152, 64), (1, 16, 40), (2, 4, 3)]:
        work = balance.kv_work_list(counts, hkv, sms, cap)
        _slices_cover(work, counts)
        lens = [s[2] for s in work["slices"]]
        seg_lens = [-(-counts[s[0]] // max(1, sum(1 for t in work["slices"] if t[0] == s[0])))
                    for s in work["slices"]]
        assert all(a >= b for a, b in zip(seg_lens[:-1], seg_lens[1:]))
        slots = sum(k - 1 for _, _, k in work["splits"])
        assert slots <= cap
        if work["L"] is not None:
            assert work["L"] >= balance.SEG_MIN
            assert max(lens) <= max(work["L"], max((c for c in counts if c <= work["L"]), default=0))


@pytest.mark.parametrize("name,cut", [("8b", False), ("70b", True), ("sparse", True),
                                      ("405b-logu", True)])
def test_kv_work_list_on_the_workloads(name, cut):
    """The rule leaves the 8B layer's lists whole (its greedy bound is within
    1.02 of the mean) and cuts the 70B shard's, the sparse-mask stress's and
    the log-uniform 405B case's, whose longest lists are several times the
    mean work per SM."""
    w = wl.WORKLOADS[name]
    cu = wl.cu_doc_lens(w)
    r = w.ranks[-1]
    c = balance.tile_counts(cu, w.batch, w.seq_len, w.cp_size, r, w.group)
    nqt = (w.seq_len // w.cp_size) // (128 // w.group)
    work = balance.kv_work_list(c["col_counts"], w.n_kv_heads, 152,
                                balance.kv_pool_slots(w.batch, w.seq_len, w.n_kv_heads, nqt))
    assert (work["L"] is not None) == cut
    _slices_cover(work, c["col_counts"].tolist())


def _greedy_makespan(lengths, sms):
    """Each item, in order, on the SM that frees first (the dK/dV kernel's
    work counter); the busiest SM's total."""
    import heapq
    free = [0] * sms
    for n in lengths:
        t = heapq.heappop(free)
        heapq.heappush(free, t + n)
    return max(free)


@pytest.mark.parametrize("name", ["70b", "sparse", "405b-logu"])
def test_kv_work_list_shortens_the_greedy_makespan(name):
    """On every rank whose lists the rule cuts, greedy scheduling of the cut
    list over 152 SMs ends no later than that of the uncut list.  It also
    stays within the list-scheduling bound of the mean plus the longest
    slice (at most L).  On the 405B shape, where the lists are long against
    the floor of 16 tiles, it ends within 1.1 x the mean, the rule's target."""
    w = wl.WORKLOADS[name]
    cu = wl.cu_doc_lens(w)
    nqt = (w.seq_len // w.cp_size) // (128 // w.group)
    cap = balance.kv_pool_slots(w.batch, w.seq_len, w.n_kv_heads, nqt)
    for r in w.ranks:
        counts = balance.tile_counts(cu, w.batch, w.seq_len, w.cp_size, r, w.group)["col_counts"]
        cut = balance.kv_work_list(counts, w.n_kv_heads, 152, cap)
        whole = balance.kv_work_list(counts, w.n_kv_heads, 152, 0)
        assert cut["L"] is not None and whole["L"] is None
        items = lambda work: [s[2] for s in work["slices"] for _ in range(w.n_kv_heads)]
        m = sum(items(cut)) / 152
        t_cut, t_whole = _greedy_makespan(items(cut), 152), _greedy_makespan(items(whole), 152)
        assert t_cut <= t_whole, (name, r)
        assert t_cut <= m + cut["L"], (name, r)
        if name.startswith("405b"):
            assert t_cut <= 1.1 * m, (name, r, t_cut / m)
