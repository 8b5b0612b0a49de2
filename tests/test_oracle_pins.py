"""Pins of the fp64 oracle to facts fixed outside it: the pages' worked block
examples and byte counts, closed forms, library routines and brute force."""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
from tests.blockpack import Q2, Q4, pack_matrix, selector_expert

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        scale, codes, weights = [s.strip() for s in line.split("|")]
        blk = bytes([int(scale[2:4], 16), int(scale[0:2], 16)]) + bytes.fromhex(codes)
        rows.append((np.frombuffer(blk, dtype=np.uint8), np.array(weights.split(), dtype=np.float64)))
    return rows


# ------------------------------------------------------------------ format

def test_f16_decode_matches_numpy_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert math.copysign(1.0, oracle.f16_to_f64(0x8000)) == -1.0


@pytest.mark.parametrize("fixture,kind,zp", [("q2_0_blocks.txt", Q2, 1), ("q4_blocks.txt", Q4, 8)])
def test_dequant_golden_blocks(fixture, kind, zp):
    rows = _read_fixture(fixture)
    assert rows
    for blk, want in rows:
        got = oracle.dequant(kind, zp, blk, want.size)
        assert np.array_equal(got, want), (fixture, got, want)
    # all blocks of the fixture decoded in one call, in order
    allb = np.concatenate([b for b, _ in rows])
    allw = np.concatenate([w for _, w in rows])
    assert np.array_equal(oracle.dequant(kind, zp, allb, allw.size), allw)


def test_q2_zero_point_two_shifts_every_weight_by_one_scale():
    # The tiny-layer configuration's Q2_0 statement uses w = d*(q-2); the page uses q-1.
    for blk, want in _read_fixture("q2_0_blocks.txt"):
        d = np.float16(0).view(np.uint16)
        d = oracle.f16_to_f64(int(blk[0]) | (int(blk[1]) << 8))
        got = oracle.dequant(Q2, 2, blk, 64)
        assert np.array_equal(got, want - d)


def test_u16_lane_order_of_the_q2_unpack():
    # "The CPU kernels": 16 code bytes are read as 8 little-endian u16 lanes; code 8i+j
    # is (lane_i >> 2j) & 3. Build lanes directly, derive bytes with numpy's '<u2' view.
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 4, size=64)
    lanes = np.zeros(8, dtype=np.uint32)
    for i in range(8):
        for j in range(8):
            lanes[i] |= int(codes[8 * i + j]) << (2 * j)
    blk = np.concatenate([np.array([0x00, 0x3C], dtype=np.uint8),
                          lanes.astype("<u2").view(np.uint8)])
    assert np.array_equal(oracle.dequant(Q2, 1, blk, 64), codes - 1.0)


def test_expert_bytes_closed_forms():
    # "The byte budget, in code": 3 x 2560 x 640 x 18 / 64 = 1,382,400 bytes; 48 layers
    # of 512 experts = the 34.0 GB arena; 10 routed experts x 48 layers = 0.66 GB/token.
    q2 = oracle.expert_bytes(Q2, 2560, 640)
    assert q2 == 1_382_400
    assert 48 * 512 * q2 == 33_973_862_400
    assert 48 * 10 * q2 == 663_552_000
    assert q2 * 8 / (3 * 2560 * 640) == 2.25  # bits per weight
    # Gemma-shaped Q4 (blocks of 32): routed 704-wide and shared 2112-wide experts
    assert oracle.expert_bytes(Q4, 2816, 704) == 3_345_408
    assert oracle.expert_bytes(Q4, 2816, 2112) == 10_036_224
    assert oracle.expert_bytes(Q4, 256, 64) == 27_648


# ------------------------------------------------------------------ router

def test_router_selector_weights_and_bias():
    rng = np.random.default_rng(1)
    T, H, E = 3, 12, 7
    x = rng.standard_normal((T, H))
    pi = rng.permutation(H)[:E]
    Wr = np.zeros((E, H))
    Wr[np.arange(E), pi] = 1.0
    b = rng.standard_normal(E)
    got = oracle.router_logits(x, Wr, b)
    assert np.array_equal(got, x[:, pi] + b)
    # a rank-1 router: every expert sees c_e * sum(x)
    c = rng.standard_normal(E)
    Wr1 = np.outer(c, np.ones(H))
    got1 = oracle.router_logits(x, Wr1)
    np.testing.assert_allclose(got1, np.outer(x.sum(1), c), rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ top-k

def _brute_topk(l, K):
    """Unique K-subset S with key(i) > key(j) for all i in S, j not in S, where
    key = (logit, -index) and NaN is below every number; S in key order."""
    E = len(l)

    def key(i):
        return (0 if np.isnan(l[i]) else 1, -np.inf if np.isnan(l[i]) else l[i], -i)

    found = []
    for S in itertools.combinations(range(E), K):
        rest = [j for j in range(E) if j not in S]
        if all(key(i) > key(j) for i in S for j in rest):
            found.append(sorted(S, key=key, reverse=True))
    assert len(found) == 1
    return found[0]


def test_topk_matches_brute_force_with_forced_ties():
    rng = np.random.default_rng(2)
    for trial in range(300):
        E = int(rng.integers(1, 11))
        K = int(rng.integers(1, E + 1))
        T = 2
        l = rng.integers(-2, 3, size=(T, E)).astype(np.float64)  # many ties
        if trial % 3 == 0:
            l += rng.standard_normal((T, E))
        if trial % 7 == 0:
            l[0, rng.integers(0, E)] = -0.0
            l[0, rng.integers(0, E)] = 0.0
        ids, w, bad = oracle.topk(l, K)
        assert not bad
        for t in range(T):
            assert list(ids[t]) == _brute_topk(l[t], K)


def test_topk_nan_ranks_last_and_flags():
    l = np.array([[1.0, np.nan, 0.5, -np.inf, 2.0]])
    ids, w, bad = oracle.topk(l, 5)
    assert bad
    assert list(ids[0]) == [4, 0, 2, 3, 1]


def test_topk_weights_are_renormalised_softmax():
    rng = np.random.default_rng(3)
    T, E = 5, 9
    l = rng.standard_normal((T, E)) * 3
    # K = 1: weight exactly 1
    ids, w, _ = oracle.topk(l, 1)
    assert np.all(w == 1.0)
    assert np.array_equal(ids[:, 0], np.argmax(l, axis=1))
    # K = E: the full softmax, in rank order
    ids, w, _ = oracle.topk(l, E)
    sm = scipy.special.softmax(l, axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(sm, ids, 1), rtol=1e-14, atol=0)
    # any K: sum 1, and w_a / w_b = exp(l_a - l_b), i.e. softmax over the selected logits
    for K in range(1, E + 1):
        ids, w, _ = oracle.topk(l, K)
        np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-15)
        sel = np.take_along_axis(l, ids, 1)
        np.testing.assert_allclose(w, scipy.special.softmax(sel, axis=1), rtol=1e-14)
        assert np.all(np.diff(sel, axis=1) <= 0)


# ------------------------------------------------------------------ bucket

@pytest.mark.parametrize("T,K,E", [(1, 1, 1), (1, 10, 512), (4, 10, 512), (4, 2, 16), (8, 8, 128),
                                   (4096, 8, 128), (3, 4, 5)])
def test_bucket_matches_stable_sort(T, K, E):
    rng = np.random.default_rng(T * 1000 + K * 10 + E)
    # top-k ids are distinct per token
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    b = oracle.bucket(ids, E)
    flat = ids.reshape(-1)
    assert np.array_equal(b["perm"], np.argsort(flat, kind="stable"))
    assert np.array_equal(b["counts"], np.bincount(flat, minlength=E))
    assert np.array_equal(b["offsets"], np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    assert np.array_equal(b["active"], np.nonzero(np.bincount(flat, minlength=E))[0])
    assert sorted(b["perm"]) == list(range(T * K))


def test_bucket_empty():
    ids = np.zeros((0, 3), dtype=np.int32)
    b = oracle.bucket(ids, 4)
    assert b["perm"].size == 0 and b["active"].size == 0
    assert np.array_equal(b["offsets"], np.zeros(5))


# ------------------------------------------------------------------ expert

def _silu(g):
    return g / (1.0 + np.exp(-g))


@pytest.mark.parametrize("kind,zp,a,b,c,dg,du,dd", [
    (Q4, 8, 9, 11, 6, 1.0, 0.5, 0.25),   # gate +1, up +3*0.5, down -2*0.25
    (Q2, 1, 2, 3, 0, 0.5, 1.0, 2.0),     # gate +1*0.5, up +2, down -1*2
    (Q2, 2, 3, 0, 1, 1.0, 0.25, 1.0),    # z = 2: gate +1, up -2*0.25, down -1
])
def test_expert_selector_pattern_closed_form(kind, zp, a, b, c, dg, du, dd):
    rng = np.random.default_rng(4)
    bw = 64 if kind == Q2 else 32
    H, F = 2 * bw, bw
    pi, sigma = rng.permutation(H)[:F], rng.permutation(H)[:F]
    rho = rng.permutation(H)[:F]
    blob = selector_expert(kind, zp, H, F, pi, sigma, rho, a, b, c, dg, du, dd)
    assert blob.size == oracle.expert_bytes(kind, H, F)
    x = rng.standard_normal((3, H))
    y = oracle.expert_ffn(kind, zp, blob, H, F, x)
    want = np.zeros_like(x)
    ga, ub, dc = dg * (a - zp), du * (b - zp), dd * (c - zp)
    want[:, rho] = dc * _silu(ga * x[:, pi]) * (ub * x[:, sigma])
    np.testing.assert_allclose(y, want, rtol=1e-14, atol=1e-14)


def test_expert_identity_pattern():
    # gate row j picks x_j, up row j picks x_j, down maps h_j to output j:
    # y_j = silu(x_j) * x_j for j < F and 0 otherwise.
    H, F = 256, 64
    idx = np.arange(F)
    blob = selector_expert(Q4, 8, H, F, idx, idx, idx, 9, 9, 9)
    x = np.random.default_rng(5).standard_normal((2, H))
    y = oracle.expert_ffn(Q4, 8, blob, H, F, x)
    want = np.zeros_like(x)
    want[:, :F] = _silu(x[:, :F]) * x[:, :F]
    np.testing.assert_allclose(y, want, rtol=1e-15, atol=1e-15)


def test_expert_gelu_tanh_closed_form():
    H, F = 64, 64
    idx = np.arange(F)
    blob = selector_expert(Q4, 8, H, F, idx, idx, idx, 9, 9, 9)
    x = np.random.default_rng(6).standard_normal((2, H))
    y = oracle.expert_ffn(Q4, 8, blob, H, F, x, act=oracle.ACT_GEGLU_TANH)
    g = x
    gelu = 0.5 * g * (1 + np.tanh(math.sqrt(2 / math.pi) * (g + 0.044715 * g ** 3)))
    np.testing.assert_allclose(y, gelu * x, rtol=1e-14, atol=1e-15)


def _identity_act(act, x):
    """act(x_j) through the oracle's expert: an identity-pattern expert (d = 1,
    gate/up/down rows select x_j) gives y_j = act(x_j) * x_j, divided back by x_j."""
    H = F = x.shape[1]
    idx = np.arange(F)
    blob = selector_expert(Q4, 8, H, F, idx, idx, idx, 9, 9, 9)
    y = oracle.expert_ffn(Q4, 8, blob, H, F, x, act=act)
    return y / x


def test_expert_activations_against_independent_implementations():
    # The activations checked against implementations written elsewhere, in fp64:
    # SiLU against scipy's logistic function (x * expit(x)), the tanh-approximated
    # GELU (Hendrycks & Gimpel's approximation, used by Gemma's experts) against
    # torch's own gelu(approximate="tanh"). A wrong constant (sqrt(pi/2) for
    # sqrt(2/pi), 0.0447 for 0.044715) or a dropped cubic term fails here.
    torch = pytest.importorskip("torch")
    from scipy.special import expit
    x = np.concatenate([np.linspace(-8, 8, 63), np.random.default_rng(61).standard_normal(65) * 3])
    x = x[np.abs(x) > 1e-3].reshape(1, -1)[:, :96]
    silu = _identity_act(oracle.ACT_SWIGLU, x)
    np.testing.assert_allclose(silu, x * expit(x), rtol=1e-13, atol=1e-300)
    gelu = _identity_act(oracle.ACT_GEGLU_TANH, x)
    want = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    np.testing.assert_allclose(gelu, want, rtol=1e-13, atol=1e-300)


def test_expert_gelu_tanh_properties():
    # Properties of the tanh form that hold whatever the constants are written as:
    # gelu(x) - gelu(-x) = x (odd part), and against the exact GELU x * Phi(x)
    # (scipy's normal CDF) the approximation's error stays below 1e-3 everywhere
    # (a wrong sqrt(2/pi) breaks this by more than 1e-2).
    from scipy.special import ndtr
    x = np.linspace(0.05, 6, 96).reshape(1, -1)
    gp, gm = _identity_act(oracle.ACT_GEGLU_TANH, x), _identity_act(oracle.ACT_GEGLU_TANH, -x)
    np.testing.assert_allclose(gp - gm, x, rtol=1e-14)
    assert np.max(np.abs(gp - x * ndtr(x))) < 1e-3


def _random_blob(rng, kind, H, F, d_lo=0.005, d_hi=0.02):
    bw = 64 if kind == Q2 else 32
    n_blocks = 3 * H * F // bw
    blk = rng.integers(0, 256, size=(n_blocks, 18)).astype(np.uint8)
    d = rng.uniform(d_lo, d_hi, size=n_blocks).astype(np.float16).view(np.uint16)
    blk[:, 0] = d & 0xFF
    blk[:, 1] = d >> 8
    return blk.reshape(-1)


def test_expert_down_scale_doubling_is_exact():
    rng = np.random.default_rng(8)
    for kind in (Q2, Q4):
        H, F = 128, 64
        blob = _random_blob(rng, kind, H, F)
        bw = 64 if kind == Q2 else 32
        nmat = H * F // bw
        blob2 = blob.copy().reshape(-1, 18)
        d = blob2[2 * nmat:, 0].astype(np.uint16) | (blob2[2 * nmat:, 1].astype(np.uint16) << 8)
        d2 = (d.view(np.float16).astype(np.float64) * 2).astype(np.float16).view(np.uint16)
        blob2[2 * nmat:, 0] = d2 & 0xFF
        blob2[2 * nmat:, 1] = d2 >> 8
        x = rng.standard_normal((2, H))
        y1 = oracle.expert_ffn(kind, 1 if kind == Q2 else 8, blob, H, F, x)
        y2 = oracle.expert_ffn(kind, 1 if kind == Q2 else 8, blob2.reshape(-1), H, F, x)
        assert np.array_equal(y2, 2 * y1)


def test_expert_matches_dense_float_reference_on_random_blob():
    # Decode the blob with numpy's float16 and bit arithmetic written independently,
    # then run the dense FFN with numpy matmuls.
    rng = np.random.default_rng(9)
    for kind, zp in ((Q2, 1), (Q4, 8)):
        H, F = 128, 64
        bw = 64 if kind == Q2 else 32
        blob = _random_blob(rng, kind, H, F)
        blk = blob.reshape(-1, 18)
        d = (blk[:, 0].astype(np.uint16) | (blk[:, 1].astype(np.uint16) << 8)).view(np.float16)
        bits = np.unpackbits(blk[:, 2:], axis=1, bitorder="little")  # bit n of the 128
        nb = 2 if kind == Q2 else 4
        q = (bits.reshape(-1, bw, nb) * (1 << np.arange(nb))).sum(-1)
        W = (d.astype(np.float64)[:, None] * (q - zp)).reshape(-1)
        Wg = W[:H * F].reshape(F, H)
        Wu = W[H * F:2 * H * F].reshape(F, H)
        Wd = W[2 * H * F:].reshape(H, F)
        x = rng.standard_normal((3, H))
        want = (_silu(x @ Wg.T) * (x @ Wu.T)) @ Wd.T
        got = oracle.expert_ffn(kind, zp, blob, H, F, x)
        np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


# ------------------------------------------------------------------ layer

def _selector_layer(kind, zp, H, E, F, rng):
    """E selector-pattern experts; expert e's down weight is (c_e - zp)."""
    bw = 64 if kind == Q2 else 32
    experts, params = [], []
    for e in range(E):
        pi, sigma, rho = rng.permutation(H)[:F], rng.permutation(H)[:F], rng.permutation(H)[:F]
        c = [0, 2, 3][e % 3] if kind == Q2 else int(rng.integers(0, 16))
        experts.append(selector_expert(kind, zp, H, F, pi, sigma, rho, zp + 1, zp + 1, c))
        params.append((pi, sigma, rho, c - zp))
    return experts, params


def _selector_out(x, p):
    pi, sigma, rho, dc = p
    y = np.zeros_like(x)
    y[..., rho] = dc * _silu(x[..., pi]) * x[..., sigma]
    return y


def test_layer_combine_closed_form_with_shared_expert():
    rng = np.random.default_rng(10)
    kind, zp, H, E, K, F = Q4, 8, 64, 6, 3, 32
    experts, params = _selector_layer(kind, zp, H, E, F, rng)
    sh_idx = rng.permutation(H)[:F]
    shared = selector_expert(kind, zp, H, F, sh_idx, sh_idx, sh_idx, 9, 9, 10)
    Wr = rng.standard_normal((E, H)) * 0.3
    bias = rng.standard_normal(E)
    x = rng.standard_normal((4, H))
    r = oracle.layer_forward(kind, zp, H, E, K, F, Wr, bias, experts, x, shared=shared, F_shared=F)
    assert r["status"] == 0
    logits = x @ Wr.T + bias
    np.testing.assert_allclose(r["logits"], logits, rtol=1e-12, atol=1e-12)
    want = np.zeros_like(x)
    for t in range(4):
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))[:K]
        assert list(r["ids"][t]) == order
        w = scipy.special.softmax(logits[t, order])
        for k, e in enumerate(order):
            want[t] += w[k] * _selector_out(x[t], params[e])
        want[t] += _selector_out(x[t], (sh_idx, sh_idx, sh_idx, 2))
    np.testing.assert_allclose(r["y"], want, rtol=1e-12, atol=1e-12)


def test_layer_top1_reproduces_the_expert_and_zero_down_leaves_shared():
    rng = np.random.default_rng(11)
    kind, zp, H, E, F = Q2, 1, 128, 4, 64
    experts = [_random_blob(rng, kind, H, F, 0.01, 0.04) for _ in range(E)]
    Wr = rng.standard_normal((E, H))
    x = rng.standard_normal((3, H))
    r = oracle.layer_forward(kind, zp, H, E, 1, F, Wr, None, experts, x)
    assert np.all(r["w"] == 1.0)
    for t in range(3):
        e = r["ids"][t, 0]
        assert np.array_equal(r["y"][t], oracle.expert_ffn(kind, zp, experts[e], H, F, x[t:t + 1])[0])
    # routed experts whose down scales are 0 contribute exactly 0: y = shared expert
    zeroed = []
    nmat = H * F // 64
    for blob in experts:
        b = blob.copy().reshape(-1, 18)
        b[2 * nmat:, 0:2] = 0
        zeroed.append(b.reshape(-1))
    shared = _random_blob(rng, kind, H, F, 0.01, 0.04)
    r2 = oracle.layer_forward(kind, zp, H, E, 2, F, Wr, None, zeroed, x, shared=shared, F_shared=F)
    assert np.array_equal(r2["y"], oracle.expert_ffn(kind, zp, shared, H, F, x))


def test_layer_token_permutation_equivariance_and_logits_in():
    rng = np.random.default_rng(12)
    kind, zp, H, E, K, F = Q4, 8, 64, 8, 2, 32
    experts = [_random_blob(rng, kind, H, F) for _ in range(E)]
    Wr = rng.standard_normal((E, H))
    x = rng.standard_normal((5, H))
    r = oracle.layer_forward(kind, zp, H, E, K, F, Wr, None, experts, x)
    p = rng.permutation(5)
    rp = oracle.layer_forward(kind, zp, H, E, K, F, Wr, None, experts, x[p])
    assert np.array_equal(rp["y"], r["y"][p])
    assert np.array_equal(rp["ids"], r["ids"][p])
    ri = oracle.layer_forward(kind, zp, H, E, K, F, None, None, experts, x, logits_in=r["logits"])
    assert np.array_equal(ri["y"], r["y"])


def test_layer_absent_expert_flags_and_contributes_nothing():
    rng = np.random.default_rng(13)
    kind, zp, H, E, K, F = Q4, 8, 64, 4, 2, 32
    experts = [_random_blob(rng, kind, H, F) for _ in range(E)]
    Wr = np.zeros((E, H))
    bias = np.array([3.0, 2.0, 1.0, 0.0])  # every token picks experts 0 and 1
    x = rng.standard_normal((2, H))
    full = oracle.layer_forward(kind, zp, H, E, K, F, Wr, bias, experts, x)
    missing = list(experts)
    missing[1] = None
    r = oracle.layer_forward(kind, zp, H, E, K, F, Wr, bias, missing, x)
    assert r["status"] == oracle.STATUS_ABSENT and full["status"] == 0
    w0 = full["w"][0, 0]
    np.testing.assert_allclose(r["y"], w0 * oracle.expert_ffn(kind, zp, experts[0], H, F, x),
                               rtol=1e-15, atol=1e-15)


# ------------------------------------------------------------------ rmsnorm

def test_rmsnorm_closed_forms():
    x = np.full((1, 8), -3.0)
    eps = 1e-6
    np.testing.assert_allclose(oracle.rmsnorm(x, eps), -1.0 / np.sqrt(1 + eps / 9.0), rtol=1e-15)
    rng = np.random.default_rng(14)
    x = rng.standard_normal((3, 100))
    y = oracle.rmsnorm(x, 0.0)
    np.testing.assert_allclose((y * y).mean(1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(oracle.rmsnorm(7.5 * x, 0.0), y, rtol=1e-14)


# ------------------------------------------------------------------ routing forms
# (kairos README "The MoE forward": per-input-dim router scale, per-expert down scale;
#  Krasis white paper sec. 5.3: sigmoid top-k; sec. 7.2-7.3: the P/M drop rule)

def _w32(*v):
    return np.array(v, dtype=np.float32)


def test_drop_rule_protects_leading_ranks_and_takes_smallest_first():
    # top-10, 75/8: ceil(10 * 75 / 100) = 8 ranks kept (the white paper's "protects
    # ranks 1-8"); ranks 9 and 10 hold 0.03 each of a total mass of 1.0
    w = _w32(0.3, 0.2, 0.1, 0.1, 0.1, 0.05, 0.05, 0.04, 0.03, 0.03)
    out, n, share, _ = oracle.route_drop(w, np.ones(10), 75, 8)
    assert n == 2 and np.array_equal(out[:8], w[:8]) and out[8] == 0 and out[9] == 0
    assert abs(share - 0.06) < 1e-6
    # 75/5: 0.03 fits, 0.06 does not; equal weights go later rank first
    out, n, share, _ = oracle.route_drop(w, np.ones(10), 75, 5)
    assert n == 1 and out[9] == 0 and out[8] == w[8] and abs(share - 0.03) < 1e-6
    # rank 10 not eligible: only rank 9 is a candidate
    el = np.ones(10)
    el[9] = 0
    out, n, _, _ = oracle.route_drop(w, el, 75, 8)
    assert n == 1 and out[8] == 0 and out[9] == w[9]


def test_drop_rule_order_is_by_weight_not_rank():
    # ranks 3 and 4 are candidates (K=4, P=50 keeps 2); rank 4 is heavier than rank 3
    w = _w32(0.5, 0.3, 0.05, 0.15)
    out, n, share, _ = oracle.route_drop(w, np.ones(4), 50, 10)
    # smallest first: 0.05 (rank 3) fits under 10%, then 0.20 > 10% stops the scan
    assert n == 1 and out[2] == 0 and out[3] == w[3] and abs(share - 0.05) < 1e-6
    # M = 100: every candidate goes (their sum never exceeds the total)
    out, n, _, _ = oracle.route_drop(w, np.ones(4), 50, 100)
    assert n == 2 and out[2] == 0 and out[3] == 0 and np.array_equal(out[:2], w[:2])


def test_drop_rule_off_cases():
    w = _w32(0.4, 0.3, 0.2, 0.1, 0.0)
    for P, M, el in [(100, 50, np.ones(5)), (0, 0, np.ones(5)), (0, 50, np.zeros(5))]:
        out, n, share, _ = oracle.route_drop(w, el, P, M)
        assert n == 0 and np.array_equal(out, w) and share == 0.0
    # a zero weight is never a candidate; P = 0 leaves every positive rank eligible
    out, n, _, _ = oracle.route_drop(w, np.ones(5), 0, 10)
    assert n == 1 and out[3] == 0 and out[4] == 0 and np.array_equal(out[:3], w[:3])


def test_drop_rule_stops_at_the_first_route_that_does_not_fit():
    # candidates ascending: 0.02, 0.05, 0.06; 10% of 1.0 admits 0.02 and 0.05 (0.07)
    # but not 0.06 (0.13); the scan stops there even though nothing smaller is left
    w = _w32(0.6, 0.27, 0.05, 0.06, 0.02)
    out, n, share, _ = oracle.route_drop(w, np.ones(5), 20, 10)
    assert n == 2 and out[4] == 0 and out[2] == 0 and out[3] == w[3] and abs(share - 0.07) < 1e-6


def test_route_weight_kinds_closed_forms():
    assert oracle.route_weights(oracle.ROUTER_SIGMOID, [0.0])[0] == 0.5
    a = 1.7
    w = oracle.route_weights(oracle.ROUTER_SIGMOID, [a, -a])
    assert abs(w[0] - 1 / (1 + math.exp(-a))) < 1e-15 and abs(w[0] + w[1] - 1.0) < 1e-15
    # sigmoid(a) + sigmoid(-a) = 1, so the normalised pair equals the plain sigmoid
    wn = oracle.route_weights(oracle.ROUTER_SIGMOID_NORM, [a, -a])
    assert np.allclose(wn, w, rtol=0, atol=1e-15)
    assert oracle.route_weights(oracle.ROUTER_SIGMOID_NORM, [0.3])[0] == 1.0
    # softmax over the K chosen = the full softmax renormalised over them (orc_topk)
    rng = np.random.default_rng(20)
    l = rng.standard_normal((1, 12))
    ids, wt, _ = oracle.topk(l, 4)
    ws = oracle.route_weights(oracle.ROUTER_SOFTMAX, l[0, ids[0]])
    np.testing.assert_allclose(ws, wt[0], rtol=1e-14, atol=1e-15)


def test_scaled_router_input():
    rng = np.random.default_rng(21)
    T, H, E = 3, 32, 5
    x = rng.standard_normal((T, H))
    Wr = rng.standard_normal((E, H))
    b = rng.standard_normal(E)
    base = oracle.router_logits(x, Wr, b)
    assert np.array_equal(oracle.router_logits_scaled(x, Wr, np.ones(H), b), base)
    two = oracle.router_logits_scaled(x, Wr, np.full(H, 2.0), b)
    np.testing.assert_allclose(two - b, 2.0 * (base - b), rtol=1e-14, atol=1e-13)
    j = 7
    onehot = np.zeros(H)
    onehot[j] = 1.0
    np.testing.assert_allclose(oracle.router_logits_scaled(x, Wr, onehot), np.outer(x[:, j], Wr[:, j]),
                               rtol=1e-15, atol=1e-15)


def test_layer_down_scale_and_router_kinds():
    rng = np.random.default_rng(22)
    kind, zp, H, E, K, F = Q4, 8, 64, 6, 3, 32
    experts, params = _selector_layer(kind, zp, H, E, F, rng)
    sh_idx = rng.permutation(H)[:F]
    shared = selector_expert(kind, zp, H, F, sh_idx, sh_idx, sh_idx, 9, 9, 10)
    Wr = rng.standard_normal((E, H)) * 0.3
    x = rng.standard_normal((4, H))
    s_e = np.array([0.5, 2.0, 0.0, 1.5, 3.0, 1.0])
    for rk in (oracle.ROUTER_SOFTMAX, oracle.ROUTER_SIGMOID, oracle.ROUTER_SIGMOID_NORM):
        r = oracle.layer_forward_routed(kind, zp, H, E, K, F, Wr, None, experts, x, shared=shared, F_shared=F,
                                        router_kind=rk, down_scale=s_e)
        assert r["status"] == 0
        logits = x @ Wr.T
        for t in range(4):
            order = sorted(range(E), key=lambda e: (-logits[t, e], e))[:K]
            assert list(r["ids"][t]) == order
            l = logits[t, order]
            if rk == oracle.ROUTER_SOFTMAX:
                w = scipy.special.softmax(l)
            else:
                w = 1 / (1 + np.exp(-l))
                if rk == oracle.ROUTER_SIGMOID_NORM:
                    w = w / w.sum()
            want = _selector_out(x[t], (sh_idx, sh_idx, sh_idx, 2))
            for k, e in enumerate(order):
                want = want + w[k] * s_e[e] * _selector_out(x[t], params[e])
            np.testing.assert_allclose(r["y"][t], want, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(r["w"][t], w * s_e[order], rtol=1e-14, atol=1e-15)


def test_layer_drop_removes_exactly_the_dropped_routes():
    rng = np.random.default_rng(23)
    kind, zp, H, E, K, F = Q4, 8, 64, 8, 4, 32
    experts, params = _selector_layer(kind, zp, H, E, F, rng)
    Wr = rng.standard_normal((E, H)) * 0.3
    x = rng.standard_normal((6, H))
    el = np.array([1, 0, 1, 1, 0, 1, 1, 1], dtype=np.uint8)
    r = oracle.layer_forward_routed(kind, zp, H, E, K, F, Wr, None, experts, x, drop_eligible=el,
                                    drop_protect_pct=50, drop_mass_pct=30)
    base = oracle.layer_forward(kind, zp, H, E, K, F, Wr, None, experts, x)
    for t in range(6):
        w32 = base["w"][t].astype(np.float32)
        want_w, n, share, _ = oracle.route_drop(w32, el[base["ids"][t]], 50, 30)
        assert r["omitted"][t] == share
        want = np.zeros(H)
        for k, e in enumerate(base["ids"][t]):
            if want_w[k] != 0:
                want += base["w"][t, k] * _selector_out(x[t], params[e])
        np.testing.assert_allclose(r["y"][t], want, rtol=1e-12, atol=1e-12)
    # the kept weights are not renormalised (softmax over the K chosen and the
    # renormalised full softmax agree to rounding)
    kept = r["w"] != 0
    assert kept.sum() < kept.size
    np.testing.assert_allclose(r["w"][kept], base["w"][kept], rtol=1e-14, atol=0)


def test_bucket_wise_layer_evaluation_equals_layer_forward():
    # the every-row prefill check evaluates the oracle one expert bucket at a time;
    # it must give the same bits as oracle.layer_forward on the same routing
    from synth import configs as C
    from tests.gpu_util import oracle_layer_by_bucket
    cfg = C.CONFIGS["gemma_layer"]
    T = 12
    x = C.as_f64(C.activations(cfg, T, step=3))
    Wr = C.as_f64(C.router_weights(cfg, 0))
    lg = (x @ Wr.T + C.router_bias(cfg, 0)).astype(np.float32)
    r = oracle_layer_by_bucket(cfg, 0, x, lg, threads=4)
    ids, _, _ = oracle.topk(lg.astype(np.float64), cfg.K)
    need = np.unique(ids)
    blobs = C.experts(cfg, 0, need)
    experts = [None] * cfg.E
    for i, e in enumerate(need):
        experts[int(e)] = blobs[i]
    r2 = oracle.layer_forward(cfg.kind, cfg.zero_point, cfg.H, cfg.E, cfg.K, cfg.F, None, None, experts, x,
                              shared=C.shared_expert(cfg, 0), F_shared=cfg.F_shared, logits_in=lg)
    assert np.array_equal(r["ids"], r2["ids"])
    assert np.array_equal(r["y"], r2["y"])
