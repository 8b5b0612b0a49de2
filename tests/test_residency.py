"""Residency policies: the reference (oracle/residency.py) pinned on hand traces, and
the library's native engine (moe_policy_*) against the reference, decision by
decision, on seeded synthetic traces. Host code only: no GPU."""
import numpy as np
import pytest

from oracle import residency as R
from quantized_expert_ffn_gb300 import _lib as L
from synth import traces


# ------------------------------------------------------------------ reference pins

def test_lru_textbook_trace():
    p = R.Policy(R.LRU, 3, 1, 8)
    out = [p.route(0, [e]) for e in (1, 2, 3, 1, 4)]
    assert [h[0] for h, _ in out] == [False, False, False, True, False]
    # 4 evicts 2: after the hit on 1, 2 is the least recently used
    assert out[4][1] == [(4, (0, 2))]
    assert p.resident == {(0, 1), (0, 3), (0, 4)}


def test_lru_never_evicts_the_event_it_serves():
    p = R.Policy(R.LRU, 2, 1, 8)
    p.route(0, [1, 2])
    hits, loads = p.route(0, [1, 2, 3])
    assert hits == [True, True, False] and loads == []  # 3 has nowhere to go
    hits, loads = p.route(0, [3, 1, 1])  # duplicates count once
    assert hits == [False, True, True] and loads == [(3, (0, 2))]


def test_decayed_frequency_scores_and_recency_guard():
    # half-life 1 token: a score halves per token
    p = R.Policy(R.DECAYED_FREQ, 2, 1, 8, half_life=1.0, guard=0)
    p.route(0, [0]); p.end_token()          # s0 = 1 at t0
    p.route(0, [0]); p.end_token()          # s0 = 1 * 0.5 + 1 = 1.5 at t1
    p.route(0, [1]); p.end_token()          # s1 = 1 at t2
    # t3: s0 = 1.5 / 4 = 0.375, s1 = 1 / 2 = 0.5 -> 0 goes
    _, loads = p.route(0, [2])
    assert loads == [(2, (0, 0))]
    # with a 2-token guard, expert 1 (used at t2) is protected at t3: 0 goes too
    q = R.Policy(R.DECAYED_FREQ, 2, 1, 8, half_life=1.0, guard=2)
    for ids in ([1], [1], [0]):
        q.route(0, ids)
        q.end_token()
    # t3: s1 = (1 * 0.5 + 1) / 4 = 0.375 < s0 = 0.5, but 0 (used at t2) is guarded
    _, loads = q.route(0, [2])
    assert loads == [(2, (0, 1))]
    q.end_token()
    # t4: s0 = 1 / 4 = 0.25, s2 = 1 / 2 = 0.5; 2 (used at t3) is guarded anyway
    _, loads = q.route(0, [3])
    assert loads == [(3, (0, 0))]


def test_lfu_swap_threshold_hysteresis_and_decay():
    p = R.Policy(R.LFU_SWAP, 2, 1, 4)
    p.seed([(0, 0), (0, 1)])
    swaps = []
    # expert 2 every token; expert 3 at tokens 2 and 4 only
    for t in range(1, 5):
        ids = [2, 3] if t % 2 == 0 else [2]
        hits, loads = p.route(0, ids)
        assert loads == []  # misses never load
        swaps.append(p.end_token())
    assert swaps[:3] == [[], [], []]
    # at the end of token 4: c2 = 1 + 0.7 + 0.49 + 0.343 = 2.533 >= 2 and beats the
    # coldest resident (expert 0, counter 0) by >= 1.5; c3 = 1 + 0.49 = 1.49 < 2
    assert swaps[3] == [(0, 2, 0)]
    assert p.resident == {(0, 1), (0, 2)}
    assert abs(float(p.cnt[(0, 2)]) - 0.7 * 2.533) < 1e-5


def test_lfu_swap_keeps_the_largest_gains_across_layers():
    p = R.Policy(R.LFU_SWAP, 2, 2, 4, swap_every=1, max_swaps=1, decay=1.0)
    p.seed([(0, 0), (1, 0)])
    for _ in range(3):
        p.route(0, [1])          # layer 0: expert 1 reaches 3 by the third token
    for _ in range(4):
        p.route(1, [2])          # layer 1: expert 2 reaches 4
    assert p.end_token() == [(1, 2, 0)]  # gain 4 beats gain 3; one swap allowed


def test_belady_textbook_trace():
    # capacity 3 over 7,0,1,2,0,3,0,4,2,3,0,3,2: the classic optimal policy has 6 hits
    seq = [7, 0, 1, 2, 0, 3, 0, 4, 2, 3, 0, 3, 2]
    events = [[(0, [e])] for e in seq]
    assert R.belady_hits(events, 3) == 6


# ------------------------------------------------------------------ engine vs reference

def _replay(kind, trace, cap, seed_pairs=None, **kw):
    T, Ln, K = trace.shape
    E = int(trace.max()) + 1
    ref = R.Policy(kind, cap, Ln, E, **kw)
    eng = L.Policy(L.policy_params(kind, cap, **{k: v for k, v in kw.items() if k != "guard"},
                                   **({"recency_guard": kw["guard"]} if "guard" in kw else {})), Ln, E)
    try:
        if seed_pairs is not None:
            n1 = ref.seed(list(zip(*seed_pairs)))
            n2 = eng.seed(*seed_pairs)
            assert n1 == n2
        hits = 0
        for t in range(T):
            for l in range(Ln):
                ids = trace[t, l]
                h_ref, loads_ref = ref.route(l, ids)
                h, le, el, ee = eng.route(l, ids)
                assert list(h.astype(bool)) == h_ref
                got = [(int(a), None if b < 0 else (int(b), int(c))) for a, b, c in zip(le, el, ee)]
                assert got == loads_ref
                for _, victim in got:  # never an expert of the event being served
                    assert victim is None or victim[0] != l or victim[1] not in ids
                hits += int(h.sum())
            sw_ref = ref.end_token()
            sw = eng.end_token()
            assert [(int(a), int(b), int(d)) for a, b, c, d in zip(*sw)] == sw_ref
            assert eng.count() == len(ref.resident) <= cap
        for l in range(Ln):
            for e in range(E):
                assert eng.resident(l, e) == ((l, e) in ref.resident)
        return hits
    finally:
        eng.close()


@pytest.mark.parametrize("seed", [1, 2])
def test_engine_matches_reference_lru(seed):
    tr = traces.routing_trace(48, 4, 48, 6, seed=seed)
    _replay(R.LRU, tr, 50)
    _replay(R.LRU, tr, 50, seed_pairs=traces.profile_ranking(tr[:8]))


@pytest.mark.parametrize("seed", [3, 4])
def test_engine_matches_reference_decayed_frequency(seed):
    tr = traces.routing_trace(48, 4, 48, 6, seed=seed)
    _replay(R.DECAYED_FREQ, tr, 50, half_life=32.0, guard=2)
    _replay(R.DECAYED_FREQ, tr, 40, half_life=4.0, guard=1, seed_pairs=traces.profile_ranking(tr[:8]))


@pytest.mark.parametrize("seed", [5, 6])
def test_engine_matches_reference_lfu_swap(seed):
    tr = traces.routing_trace(64, 4, 48, 6, seed=seed)
    _replay(R.LFU_SWAP, tr, 60, seed_pairs=traces.profile_ranking(tr[:8]))
    _replay(R.LFU_SWAP, tr, 60, seed_pairs=traces.profile_ranking(tr[:4]), max_swaps=3, swap_every=2)


@pytest.mark.parametrize("half_life,guard,cap,seeded", [(1.0, 0, 3, False), (1.0, 2, 4, True), (0.5, 1, 5, True),
                                                        (4.0, 0, 6, False), (1000.0, 2, 7, True)])
def test_engine_matches_reference_decayed_frequency_on_ties(half_life, guard, cap, seeded):
    # few experts and short or very long half-lives: many pairs share a history, so
    # decayed scores tie exactly and the recency and pair-index tie-breaks decide
    tr = traces.routing_trace(160, 2, 8, 3, seed=int(half_life * 10) + cap, zipf_s=0.3, stick=0.2)
    prof = traces.profile_ranking(tr[:5]) if seeded else None
    _replay(R.DECAYED_FREQ, tr, cap, seed_pairs=prof, half_life=half_life, guard=guard)


@pytest.mark.parametrize("guard,cap,seeded", [(8, 60, False), (16, 60, True), (16, 120, True)])
def test_engine_matches_reference_decayed_frequency_long_guard(guard, cap, seeded):
    # long recency guards keep many pairs outside the victim heap at once (held until
    # their guard ends, released in order, the heap rebuilt with them); pools large
    # enough that the heap, not the fallback scan, picks most victims
    tr = traces.routing_trace(120, 4, 64, 6, seed=guard * 7 + cap)
    prof = traces.profile_ranking(tr[:8]) if seeded else None
    _replay(R.DECAYED_FREQ, tr, cap, seed_pairs=prof, half_life=32.0, guard=guard)


def test_seed_checks_every_pair_before_placing_any():
    p = L.Policy(L.policy_params(L.POLICY_DECAYED_FREQ, 8), 2, 8)
    try:
        with pytest.raises(L.MoeError):
            p.seed([0, 1, 5], [1, 2, 3])  # the third pair's layer is out of range
        assert p.count() == 0
        with pytest.raises(L.MoeError):
            p.seed([0, 1], [1, 8])  # expert out of range
        assert p.count() == 0
        assert p.seed([0, 1], [1, 2]) == 2
        assert p.count() == 2
    finally:
        p.close()


def test_hit_rates_are_bounded_by_belady():
    tr = traces.routing_trace(64, 4, 64, 8, seed=7)
    events = [[(l, tr[t, l]) for l in range(4)] for t in range(64)]
    prof = traces.profile_ranking(tr[:8])
    bel = R.belady_hits(events, 80, list(zip(*prof)))
    for kind in (R.LRU, R.DECAYED_FREQ):
        assert _replay(kind, tr, 80, seed_pairs=prof) <= bel


def test_policy_argument_checks():
    with pytest.raises(L.MoeError):
        L.Policy(L.policy_params(7, 10), 2, 8)
    with pytest.raises(L.MoeError):
        L.Policy(L.policy_params(L.POLICY_LRU, 0), 2, 8)
    p = L.Policy(L.policy_params(L.POLICY_LRU, 4), 2, 8)
    try:
        with pytest.raises(L.MoeError):
            p.route(2, [0])
        with pytest.raises(L.MoeError):
            p.route(0, [8])
    finally:
        p.close()


@pytest.mark.parametrize("seed,cap", [(8, 40), (9, 100), (10, 7)])
def test_engine_belady_matches_reference(seed, cap):
    tr = traces.routing_trace(40, 3, 40, 6, seed=seed)
    prof = traces.profile_ranking(tr[:6])
    events = [[(l, tr[t, l]) for l in range(3)] for t in range(40)]
    assert L.moe_policy_belady(tr, 40, cap, *prof) == R.belady_hits(events, cap, list(zip(*prof)))
    assert L.moe_policy_belady(tr, 40, cap) == R.belady_hits(events, cap)
    seq = np.array([7, 0, 1, 2, 0, 3, 0, 4, 2, 3, 0, 3, 2], dtype=np.int32).reshape(-1, 1, 1)
    assert L.moe_policy_belady(seq, 8, 3) == 6


# ------------------------------------------------------------------ a whole token per call

@pytest.mark.parametrize("kind,kw", [(L.POLICY_LRU, {}), (L.POLICY_DECAYED_FREQ, {"half_life": 4.0}),
                                     (L.POLICY_DECAYED_FREQ, {"half_life": 1.0, "recency_guard": 0}),
                                     (L.POLICY_LFU_SWAP, {"swap_every": 2, "max_swaps": 5})])
@pytest.mark.parametrize("seeded", [False, True])
def test_route_token_equals_per_layer_routes(kind, kw, seeded):
    tr = traces.routing_trace(40, 6, 24, 4, seed=21 + kind)
    a = L.Policy(L.policy_params(kind, 30, **kw), 6, 24)
    b = L.Policy(L.policy_params(kind, 30, **kw), 6, 24)
    try:
        if seeded:
            prof = traces.profile_ranking(tr[:5])
            assert a.seed(*prof) == b.seed(*prof)
        for t in range(40):
            hits, plan = [], [[], [], [], []]
            for l in range(6):
                h, le, el, ee = a.route(l, tr[t, l])
                hits.append(h)
                for lst, vals in zip(plan, (np.full(le.size, l, np.int32), le, el, ee)):
                    lst.extend(int(v) for v in vals)
            hb, ll, le, el, ee = b.route_token(tr[t])
            assert np.array_equal(hb, np.stack(hits))
            assert [list(map(int, x)) for x in (ll, le, el, ee)] == plan
            sa, sb = a.end_token(), b.end_token()
            assert all(np.array_equal(x, y) for x, y in zip(sa, sb))
        assert a.count() == b.count()
        assert all(a.resident(l, e) == b.resident(l, e) for l in range(6) for e in range(24))
    finally:
        a.close()
        b.close()


def test_route_token_checks_before_changing_anything():
    p = L.Policy(L.policy_params(L.POLICY_LRU, 8), 3, 16)
    try:
        p.route_token(np.array([[0, 1], [2, 3], [4, 5]], dtype=np.int32))
        assert p.count() == 6
        bad = np.array([[6, 7], [8, 9], [10, 16]], dtype=np.int32)  # the last id is out of range
        with pytest.raises(L.MoeError):
            p.route_token(bad)
        assert p.count() == 6 and not p.resident(0, 6)
        with pytest.raises(L.MoeError):
            p.route_token(np.zeros((4, 2), dtype=np.int32))  # more layers than the policy has
        ids = np.array([[6, 7]], dtype=np.int32)
        hit = np.zeros((1, 2), np.uint8)
        short = [np.zeros(1, np.int32) for _ in range(4)]
        with pytest.raises(L.MoeError):
            L.moe_policy_route_token(p.h, ids, hit, *short, 1)  # cap below n_layers * K
        assert p.count() == 6
        hit, ll, le, el, ee = p.route_token(np.zeros((0, 2), dtype=np.int32))
        assert hit.shape == (0, 2) and ll.size == 0 and p.count() == 6
    finally:
        p.close()
