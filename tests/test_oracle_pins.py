"""Pins for the CPU oracle against what the pages and the mathematics fix.

None of these checks re-types the oracle's own formula: each one compares it with
a hand-worked value (tests/golden), a closed form, a library routine, a brute
force, or an invariant that a dropped term, wrong sign, wrong index or transposed
operand would break.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------- fp16

def test_half_conversion_matches_numpy():
    vals = np.array([0.0, -0.0, 1.0, -2.5, 65504.0, 1e-8, 2.0 ** -24, 0.1, 1 + 2.0 ** -11,
                     1 + 3 * 2.0 ** -11, 3.14159, -0.0123, 70000.0], np.float32)
    for v in vals:
        assert oracle.float_to_half(v) == int(np.float16(v).view(np.uint16)), v
    for h in [0x0000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0xC400, 0x2E66, 0x8001]:
        assert oracle.half_to_double(h) == float(np.uint16(h).view(np.float16))


# ----------------------------------------------------------------- dequant

def _group_words(case):
    bits, K = case["bits"], case["K"]
    nw = K * bits // 32
    if case.get("fill"):
        return np.array([int(case["words"][0], 16)] * nw, np.uint32)
    if case.get("fill_pattern"):
        return np.array([(4 * i) | (4 * i + 1) << 8 | (4 * i + 2) << 16 | (4 * i + 3) << 24
                         for i in range(nw)], np.uint32)
    return np.array([int(w, 16) for w in case["words"]], np.uint32)


@pytest.mark.parametrize("case", _load("affine_groups.json")["cases"], ids=lambda c: c["name"])
def test_dequant_hand_built_groups(case):
    bits, K = case["bits"], case["K"]
    q = _group_words(case)[None, :]
    s = np.array([[int(case["scale_f16"], 16)]], np.uint16)
    b = np.array([[int(case["bias_f16"], 16)]], np.uint16)
    w = oracle.dequant(q, s, b, K, bits)[0]
    if "expect_all" in case:
        assert np.all(w == case["expect_all"])
    if "expect_first16" in case:
        assert list(w[:16]) == case["expect_first16"]
        assert list(w[16:32]) == case["expect_first16"]
    if "expect_first8" in case:
        assert list(w[:8]) == case["expect_first8"]
        assert list(w) == [1.0 + 0.25 * j for j in range(64)]
    if case["name"] == "one_hot4_col37":
        exp = np.zeros(64)
        exp[37] = 18.0
        assert np.array_equal(w, exp)


def test_dequant_group_boundaries_use_their_own_scale():
    # two groups, same codes, different scale/bias: the second half must use group 1's pair
    K = 128
    q = np.full((1, K // 8), 0x11111111, np.uint32)  # every code 1
    s = np.array([[0x3C00, 0x4000]], np.uint16)  # 1.0, 2.0
    b = np.array([[0x0000, 0x3C00]], np.uint16)  # 0.0, 1.0
    w = oracle.dequant(q, s, b, K, 4)[0]
    assert np.all(w[:64] == 1.0) and np.all(w[64:] == 3.0)


# ----------------------------------------------------------------- quantiser

def test_quantise_recovers_codes_on_the_grid():
    rng = np.random.default_rng(1)
    N, K = 8, 256
    codes = rng.integers(0, 16, (N, K))
    codes[:, ::64] = 0   # make min and max of every group hit the code range ends
    codes[:, 1::64] = 15
    w = (0.25 * codes - 1.5).astype(np.float32)
    q, s, b = oracle.quantise(w, 4)
    assert np.all(s == 0x3400) and np.all(b == 0xBE00)  # 0.25, -1.5
    assert np.array_equal(oracle.dequant(q, s, b, K, 4), w.astype(np.float64))


def test_quantise_nibble_layout():
    w = np.tile(np.arange(16, dtype=np.float32), 4)[None, :]  # codes 0..15 with s=1, b=0
    q, s, b = oracle.quantise(w, 4)
    assert list(q[0]) == [0x76543210, 0xFEDCBA98] * 4
    w8 = np.arange(64, dtype=np.float32)[None, :] * 4.0  # 8-bit: max 252 -> s = 252/255
    q8, s8, b8 = oracle.quantise(w8, 8)
    assert b8[0, 0] == 0
    assert q8[0, 0] & 0xFF == 0 and (q8[0, 15] >> 24) == 255


def test_quantise_error_bound_and_constant_group():
    rng = np.random.default_rng(2)
    w = (rng.standard_normal((16, 512)) * 0.02).astype(np.float32)
    w[3, 64:128] = 0.0123  # constant group -> scale 0, code 0, bias = value
    for bits in (4, 8):
        q, s, b = oracle.quantise(w, bits)
        d = oracle.dequant(q, s, b, 512, bits)
        sf = s.astype(np.uint16).view(np.float16).astype(np.float64).repeat(64, axis=1)
        bf = b.astype(np.uint16).view(np.float16).astype(np.float64).repeat(64, axis=1)
        # half a step plus the fp16 rounding of the bias (2^-11 relative) plus slack
        bound = 0.5 * sf + np.abs(bf) * 2.0 ** -11 + 1e-7
        assert np.all(np.abs(d - w) <= bound + sf * 1e-3)
        assert s[3, 1] == 0 and b[3, 1] == np.float16(0.0123).view(np.uint16)
        assert np.all(d[3, 64:128] == float(np.float16(0.0123)))


# ----------------------------------------------------------------- qgemv

def test_qgemv_permutation_matrix_is_exact():
    # row n selects column perm[n] (code 1, scale 1, bias 0): y = x[perm] exactly.
    N, K = 96, 128
    rng = np.random.default_rng(3)
    perm = rng.permutation(K)[:N]
    q = np.zeros((N, K // 8), np.uint32)
    for n, c in enumerate(perm):
        q[n, c // 8] |= np.uint32(1 << (4 * (c % 8)))
    s = np.full((N, K // 64), 0x3C00, np.uint16)
    b = np.zeros((N, K // 64), np.uint16)
    x = rng.standard_normal((3, K)).astype(np.float32)
    y = oracle.qgemv(q, s, b, K, 4, x)
    assert np.array_equal(y, x[:, perm].astype(np.float64))


def test_qgemv_constant_codes_closed_form():
    # every code c, scale s_g, bias b_g: y = sum_g (s_g c + b_g) * sum_{j in g} x_j
    N, K = 4, 192
    q = np.full((N, K // 8), 0x55555555, np.uint32)  # code 5
    s = np.array([[0x3800, 0x3C00, 0x4000]] * N, np.uint16)  # 0.5, 1, 2
    b = np.array([[0x0000, 0xBC00, 0x3800]] * N, np.uint16)  # 0, -1, 0.5
    x = np.arange(K, dtype=np.float32) / 7.0
    xs = [float(np.sum(x[g * 64:(g + 1) * 64].astype(np.float64))) for g in range(3)]
    expect = (0.5 * 5 + 0) * xs[0] + (1 * 5 - 1) * xs[1] + (2 * 5 + 0.5) * xs[2]
    y = oracle.qgemv(q, s, b, K, 4, x)
    assert np.allclose(y, expect, rtol=1e-13)


def test_qgemv_matches_library_matmul():
    rng = np.random.default_rng(4)
    N, K = 64, 320
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    for bits in (4, 8):
        q, s, b = oracle.quantise(w, bits)
        x = rng.standard_normal((5, K)).astype(np.float32)
        y = oracle.qgemv(q, s, b, K, bits, x)
        ref = x.astype(np.float64) @ oracle.dequant(q, s, b, K, bits).T
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------- routing

def _identity_router(E, H):
    """Router whose logit e is x[e] exactly (8-bit code 1 at column e, scale 1, bias 0)."""
    q = np.zeros((E, H // 4), np.uint32)
    for e in range(E):
        q[e, e // 4] |= np.uint32(1 << (8 * (e % 4)))
    s = np.full((E, H // 64), 0x3C00, np.uint16)
    b = np.zeros((E, H // 64), np.uint16)
    return q, s, b


def _brute_topk(l, k):
    """The unique k-subset whose every member outranks every non-member, ranked by
    (value desc, index asc); returned in rank order."""
    E = len(l)
    key = lambda e: (l[e], -e)
    for sub in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in sub]
        if all(key(a) > key(r) for a in sub for r in rest):
            return sorted(sub, key=key, reverse=True)
    raise AssertionError("no top-k subset")


@pytest.mark.parametrize("E,k", [(8, 8), (10, 3), (12, 8), (12, 1), (11, 5)])
def test_topk_brute_force_with_ties(E, k):
    H = 64
    rq, rs, rb = _identity_router(E, H)
    rng = np.random.default_rng(E * 100 + k)
    for trial in range(30):
        x = np.zeros(H, np.float32)
        # small integer values force plenty of exact ties
        x[:E] = rng.integers(-3, 4, E).astype(np.float32)
        if trial % 3 == 0:
            x[:E] = rng.standard_normal(E).astype(np.float32)
        _, idx, gate = oracle.route(rq, rs, rb, E, H, x, topk=k)
        assert list(idx[0]) == _brute_topk([float(v) for v in x[:E]], k)
        assert abs(gate[0].sum() - 1.0) < 1e-12


def test_all_equal_logits_pick_lowest_indices_and_equal_gates():
    E, H = 32, 64
    rq, rs, rb = _identity_router(E, H)
    _, idx, gate = oracle.route(rq, rs, rb, E, H, np.zeros(H, np.float32), topk=8)
    assert list(idx[0]) == list(range(8))
    assert np.all(gate[0] == 0.125)


def test_two_expert_gate_closed_form_and_bias():
    E, H = 4, 64
    rq, rs, rb = _identity_router(E, H)
    x = np.zeros(H, np.float32)
    x[:4] = [0.5, 2.0, -1.0, 1.25]
    bias = np.array([0.0, -3.0, 0.0, 0.0], np.float32)  # expert 1: 2.0 - 3.0 = -1.0
    logits, idx, gate = oracle.route(rq, rs, rb, E, H, x, topk=2, logit_bias=bias)
    assert list(logits[0]) == [0.5, -1.0, -1.0, 1.25]
    assert list(idx[0]) == [3, 0]
    assert abs(gate[0, 0] - 1.0 / (1.0 + math.exp(0.5 - 1.25))) < 1e-15
    assert abs(gate[0, 1] - 1.0 / (1.0 + math.exp(1.25 - 0.5))) < 1e-15


# ----------------------------------------------------------------- GeGLU / expert

def test_gelu_tanh_library_and_normal_cdf():
    import torch
    import torch.nn.functional as F
    from scipy.special import ndtr
    zs = [-4.0, -1.0, -0.3, 0.0, 0.5, 1.0, 2.0, 3.7]
    lib = F.gelu(torch.tensor(zs, dtype=torch.float64), approximate="tanh").tolist()
    for z, v in zip(zs, lib):
        assert abs(oracle.gelu_tanh(z) - v) < 1e-15
        # the tanh form tracks the exact z * Phi(z) to about 1e-3
        assert abs(oracle.gelu_tanh(z) - z * ndtr(z)) < 1e-3
    assert abs(oracle.gelu_tanh(1.0) - 0.8411919906082768) < 1e-15


def _onehot_rows(rows, K, cols, code=1):
    q = np.zeros((rows, K // 8), np.uint32)
    for r, c in enumerate(cols):
        q[r, c // 8] |= np.uint32(code << (4 * (c % 8)))
    return q


def test_expert_geglu_and_down_orientation():
    """gate row i and up row i both pick x[i]; down row n picks h[(5n+1) mod I]:
    out[n] = gelu(x_m) x_m with m = (5n+1) mod I.  A swapped gate/up, a missing
    product, or a transposed down matrix all change the answer."""
    H, I = 128, 64
    one = lambda r, K: np.full((r, K // 64), 0x3C00, np.uint16)
    zero = lambda r, K: np.zeros((r, K // 64), np.uint16)
    gate_cols = list(range(I))
    up_cols = list(range(I))
    gu_q = np.concatenate([_onehot_rows(I, H, gate_cols), _onehot_rows(I, H, up_cols, code=2)])
    gu_s, gu_b = one(2 * I, H), zero(2 * I, H)
    dcols = [(5 * n + 1) % I for n in range(H)]
    d_q = _onehot_rows(H, I, dcols)
    blob = oracle.pack_expert(H, I, (gu_q, gu_s, gu_b), (d_q, one(H, I), zero(H, I)))
    x = np.linspace(-2.5, 2.5, H).astype(np.float32)
    out, h = oracle.expert(blob, H, I, x)
    for i in range(I):
        xi = float(x[i])
        assert abs(h[i] - oracle.gelu_tanh(xi) * 2.0 * xi) < 1e-15
    for n in range(H):
        assert out[n] == h[dcols[n]]


# ----------------------------------------------------------------- the layer

def _random_blob(rng, H, I, scale_down=1.0):
    gu = (rng.standard_normal((2 * I, H)) * 0.02).astype(np.float32)
    d = (rng.standard_normal((H, I)) * 0.02 * scale_down).astype(np.float32)
    return oracle.pack_expert(H, I, oracle.quantise(gu, 4), oracle.quantise(d, 4))


def _small_layer(seed=5, H=128, E=12, I=64, Is=128):
    rng = np.random.default_rng(seed)
    router = oracle.quantise((rng.standard_normal((E, H)) * 0.3).astype(np.float32), 8)
    experts = [_random_blob(rng, H, I) for _ in range(E)]
    shared = _random_blob(rng, H, Is)
    x = rng.standard_normal((4, H)).astype(np.float32)
    return H, E, I, Is, router, experts, shared, x


def test_layer_identical_experts_is_routing_independent():
    H, E, I, Is, router, experts, shared, x = _small_layer()
    same = [experts[0]] * E
    y1, idx1, _ = oracle.moe_layer(H, E, 8, I, Is, router, same, shared, x)
    bias = np.zeros(E, np.float32)
    bias[:4] = -50.0  # forces a different top-8
    y2, idx2, _ = oracle.moe_layer(H, E, 8, I, Is, router, same, shared, x, logit_bias=bias)
    assert not np.array_equal(np.sort(idx1, axis=1), np.sort(idx2, axis=1))
    assert np.allclose(y1, y2, rtol=1e-12, atol=1e-13)
    # and equals one expert plus the shared expert (gates sum to one)
    for t in range(x.shape[0]):
        o, _ = oracle.expert(experts[0], H, I, x[t])
        s, _ = oracle.expert(shared, H, Is, x[t])
        assert np.allclose(y1[t], o + s, rtol=1e-12, atol=1e-13)


def test_layer_is_gate_weighted_sum_plus_shared():
    H, E, I, Is, router, experts, shared, x = _small_layer(seed=6)
    y, idx, gate = oracle.moe_layer(H, E, 8, I, Is, router, experts, shared, x)
    _, ridx, rgate = oracle.route(*router, E, H, x, topk=8)
    assert np.array_equal(idx, ridx) and np.array_equal(gate, rgate)
    for t in range(x.shape[0]):
        acc = np.zeros(H)
        for k in range(8):
            acc += gate[t, k] * oracle.expert(experts[idx[t, k]], H, I, x[t])[0]
        acc += oracle.expert(shared, H, Is, x[t])[0]
        assert np.array_equal(acc, y[t])


def test_layer_down_scale_doubling_doubles_routed_part():
    H, E, I, Is, router, experts, shared, x = _small_layer(seed=7)
    off = oracle.expert_blob_offsets(H, I)
    doubled = []
    for bl in experts:
        bl = bl.copy()
        for part in (4, 5):  # down scales and biases, fp16: x2 is exact
            a = bl[off[part]:off[part] + H * (I // 64) * 2].view(np.uint16)
            a[:] = (a.view(np.float16).astype(np.float32) * 2).astype(np.float16).view(np.uint16)
        doubled.append(bl)
    y1, _, _ = oracle.moe_layer(H, E, 8, I, Is, router, experts, shared, x)
    y2, _, _ = oracle.moe_layer(H, E, 8, I, Is, router, doubled, shared, x)
    ys = np.stack([oracle.expert(shared, H, Is, x[t])[0] for t in range(x.shape[0])])
    assert np.allclose(y2 - ys, 2 * (y1 - ys), rtol=1e-11, atol=1e-13)


def test_layer_expert_permutation_equivariance():
    H, E, I, Is, router, experts, shared, x = _small_layer(seed=8)
    perm = np.random.default_rng(0).permutation(E)  # new expert p holds old expert perm[p]
    rq, rs, rb = router
    router_p = (rq[perm], rs[perm], rb[perm])
    experts_p = [experts[perm[p]] for p in range(E)]
    y1, idx1, g1 = oracle.moe_layer(H, E, 8, I, Is, router, experts, shared, x)
    y2, idx2, g2 = oracle.moe_layer(H, E, 8, I, Is, router_p, experts_p, shared, x)
    assert np.array_equal(perm[idx2], idx1)
    assert np.array_equal(y1, y2) and np.array_equal(g1, g2)


def test_layer_batch_equals_single_tokens_and_residual():
    H, E, I, Is, router, experts, shared, x = _small_layer(seed=9)
    yb, idxb, gb = oracle.moe_layer(H, E, 8, I, Is, router, experts, shared, x)
    for t in range(x.shape[0]):
        y1, i1, g1 = oracle.moe_layer(H, E, 8, I, Is, router, experts, shared, x[t:t + 1])
        assert np.array_equal(y1[0], yb[t]) and np.array_equal(i1[0], idxb[t])
    yr, _, _ = oracle.moe_layer(H, E, 8, I, Is, router, experts, shared, x, residual=True)
    assert np.array_equal(yr, yb + x.astype(np.float64))


def test_layer_rejects_missing_routed_expert():
    H, E, I, Is, router, experts, shared, x = _small_layer(seed=10)
    _, idx, _ = oracle.route(*router, E, H, x[:1], topk=8)
    holes = list(experts)
    holes[idx[0, 3]] = None
    with pytest.raises(ValueError):
        oracle.moe_layer(H, E, 8, I, Is, router, holes, shared, x[:1])


# ----------------------------------------------------------------- RMSNorm

def test_rmsnorm_hand_worked_rows():
    # x = (3, 4): mean of squares 12.5, rms = sqrt(12.5) = 5 / sqrt(2)
    #   -> (3, 4) * sqrt(2) / 5 = (0.848528137..., 1.131370849...)
    out = oracle.rmsnorm(np.array([3.0, 4.0], np.float32), np.ones(2, np.float32), 0.0)
    assert np.allclose(out, [3 * math.sqrt(2) / 5, 4 * math.sqrt(2) / 5], rtol=1e-15, atol=0)
    # one-hot 3 e_1 in H = 4: mean of squares 9/4, rms 1.5 -> 2 g_1 at index 1, 0 elsewhere
    g = np.array([0.5, -1.25, 2.0, 3.0], np.float32)
    out = oracle.rmsnorm(np.array([0.0, 3.0, 0.0, 0.0], np.float32), g, 0.0)
    assert np.array_equal(out, [0.0, 2 * -1.25, 0.0, 0.0])
    # a constant row c with eps: g c / sqrt(c^2 + eps) (c = 2, eps = 0.25 -> g 2 / sqrt(4.25))
    out = oracle.rmsnorm(np.full(8, 2.0, np.float32), np.arange(8, dtype=np.float32), 0.25)
    assert np.allclose(out, np.arange(8) * 2 / math.sqrt(4.25), rtol=1e-15, atol=0)
    # a zero row stays zero (eps > 0: no division by zero)
    assert np.array_equal(oracle.rmsnorm(np.zeros((2, 5), np.float32), np.ones(5, np.float32), 1e-6),
                          np.zeros((2, 5)))


def test_rmsnorm_invariants():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 96)).astype(np.float32)
    g = np.ones(96, np.float32)
    out = oracle.rmsnorm(x, g, 0.0)
    # unit root mean square per row when g = 1 and eps = 0
    assert np.allclose(np.sqrt(np.mean(out ** 2, axis=1)), 1.0, rtol=1e-14)
    # scale invariance (eps = 0): a power-of-two scale is exact in fp32
    assert np.allclose(oracle.rmsnorm(x * np.float32(8.0), g, 0.0), out, rtol=1e-14)
    # rows are independent, and g multiplies elementwise
    g2 = rng.standard_normal(96).astype(np.float32)
    assert np.allclose(oracle.rmsnorm(x, g2, 0.0), out * g2.astype(np.float64), rtol=1e-14)
    assert np.array_equal(oracle.rmsnorm(x[1], g2, 1e-5), oracle.rmsnorm(x, g2, 1e-5)[1])


def test_prenorm_block_is_residual_plus_layer_of_normalised_input():
    H, E, I, Is, router, experts, shared, x = _small_layer(seed=12)
    g = np.linspace(0.5, 1.5, H).astype(np.float32)
    yb, ib, gb = oracle.moe_block(H, E, 8, I, Is, router, experts, shared, x, g, 1e-6)
    xn = oracle.rmsnorm(x, g, 1e-6).astype(np.float32)
    yl, il, gl = oracle.moe_layer(H, E, 8, I, Is, router, experts, shared, xn)
    assert np.array_equal(ib, il) and np.array_equal(gb, gl)
    assert np.array_equal(yb, yl + x.astype(np.float64))
    # the layer sees a normalised input: scaling x by 4 changes only the residual
    y4, i4, _ = oracle.moe_block(H, E, 8, I, Is, router, experts, shared, x * np.float32(4.0), g, 0.0)
    y1, i1, _ = oracle.moe_block(H, E, 8, I, Is, router, experts, shared, x, g, 0.0)
    assert np.array_equal(i4, i1)
    assert np.allclose(y4 - 4 * x.astype(np.float64), y1 - x.astype(np.float64), rtol=1e-6, atol=1e-9)


# ----------------------------------------------------------------- sampling

def test_sample_hand_worked():
    # logits (1, 3, 2, 3, 0.5), temperature 1, top-K 3: the kept tokens in order are
    # 1, 3 (tie with 1: the lower index first), 2 with weights 1, 1, e^-1; totals
    # 1, 2, 2 + e^-1 = 2.3679
    lg = [1.0, 3.0, 2.0, 3.0, 0.5]
    e1 = math.exp(-1.0)
    total = 2.0 + e1
    # top-P 0.9: the cumulative 1/total, 2/total (0.845) stay below, so all three stay
    assert oracle.sample(lg, 1.0, 3, 0.9, 0.2)[0] == 1          # 0.2 * total < 1
    assert oracle.sample(lg, 1.0, 3, 0.9, 0.5)[0] == 3          # 1 <= 0.5 * total < 2
    assert oracle.sample(lg, 1.0, 3, 0.9, 0.9)[0] == 2          # 0.9 * total >= 2
    # top-P 0.8: 2 / total = 0.845 reaches it, so tokens 1 and 3 remain (total 2)
    assert oracle.sample(lg, 1.0, 3, 0.8, 0.9)[0] == 3          # 0.9 * 2 = 1.8 < 2
    assert oracle.sample(lg, 1.0, 3, 0.8, 0.45)[0] == 1         # 0.9 < 1
    # the margin of u = 0.5 with top-P 0.9 is the top-P decision: |2 / total - 0.9|
    assert abs(oracle.sample(lg, 1.0, 3, 0.9, 0.5)[1] - abs(2 / total - 0.9)) < 1e-12


def test_sample_greedy_and_degenerate_cuts():
    rng = np.random.default_rng(7)
    lg = rng.standard_normal(300).astype(np.float32)
    lg[[17, 250]] = 9.0  # tied maximum: the lower index wins
    for u in (0.0, 0.3, 0.999):
        assert oracle.sample(lg, 0.0, 64, 0.95, u)[0] == 17     # greedy
        assert oracle.sample(lg, 0.7, 1, 0.95, u)[0] == 17      # top-K 1
        assert oracle.sample(lg, 0.7, 64, 1e-9, u)[0] == 17     # top-P keeps one token
    # a power-of-two temperature is a power-of-two rescaling of the logits
    for u in (0.1, 0.6, 0.95):
        assert oracle.sample(lg, 2.0, 50, 0.9, u)[0] == oracle.sample(lg / np.float32(2.0), 1.0, 50, 0.9, u)[0]


def test_sample_frequencies_are_the_softmax():
    # no cuts: over a uniform grid of u, token j is drawn for a share of the grid equal
    # to its softmax probability (to within one grid step per boundary)
    lg = np.array([0.3, -1.2, 2.0, 0.0, 1.1, -0.4, 0.9], np.float32)
    temp = 0.8
    n = 20000
    counts = np.zeros(lg.size)
    for k in range(n):
        counts[oracle.sample(lg, temp, 0, 1.0, (k + 0.5) / n)[0]] += 1
    z = lg.astype(np.float64) / temp
    p = np.exp(z - z.max())
    p /= p.sum()
    assert np.all(np.abs(counts / n - p) <= 2.0 / n)


# ----------------------------------------------------------------- LFU

def _lfu_cases():
    return {c["name"]: c for c in _load("lfu_traces.json")["cases"]}


def test_lfu_hand_trace():
    c = _lfu_cases()["fill_hit_evict_ties"]
    lfu = oracle.LFU(c["slots"], c["E"])
    for st in c["steps"]:
        slot, hit = lfu.step(st["req"])
        assert list(slot) == st["slot"] and list(hit.astype(int)) == st["hit"], st
    eos, cnt, last, hits, misses = lfu.state()
    f = c["final"]
    assert list(eos) == f["expert_of_slot"] and list(cnt) == f["count"]
    assert list(last) == f["last"] and (hits, misses) == (f["hits"], f["misses"])


def test_lfu_seventeen_cyclic_thrash():
    c = _lfu_cases()["seventeen_cyclic_thrash"]
    lfu = oracle.LFU(c["slots"], c["E"])
    for s in range(c["cyclic"]["steps"]):
        slot, hit = lfu.step([s % c["cyclic"]["period"]])
        assert not hit[0] and slot[0] == s % 16
    assert lfu.state()[3:] == (c["hits"], c["misses"])


def test_lfu_hot_set_stays():
    c = _lfu_cases()["hot_eight_never_evicted"]
    lfu = oracle.LFU(c["slots"], c["E"])
    for s in range(c["steps"]):
        req = c["hot"] + [c["cold_base"] + s % c["cold_count"]]
        slot, hit = lfu.step(req)
        assert list(slot[:8]) == c["hot_slots"]
        assert bool(hit[8]) is False
        assert all(hit[:8]) == (s > 0)
    assert lfu.state()[3:] == (c["hits"], c["misses"])


def test_lfu_rejects_bad_requests_without_change():
    lfu = oracle.LFU(4, 10)
    lfu.step([1, 2])
    before = [a.copy() if hasattr(a, "copy") else a for a in lfu.state()]
    with pytest.raises(ValueError):
        lfu.step([3, 3])
    with pytest.raises(ValueError):
        lfu.step([10])
    with pytest.raises(ValueError):
        lfu.step([-1])
    with pytest.raises(OverflowError):
        lfu.step([0, 1, 2, 3, 4])
    after = lfu.state()
    for a, b in zip(before, after):
        assert np.array_equal(a, b)


# ----------------------------------------------------------------- tile layout

def _mlx_parts(blob, H, I):
    off = oracle.expert_blob_offsets(H, I)
    sizes = [2 * I * H // 2, 2 * I * (H // 64) * 2, 2 * I * (H // 64) * 2, H * I // 2,
             H * (I // 64) * 2, H * (I // 64) * 2]
    shapes = [(2 * I, H // 8), (2 * I, H // 64), (2 * I, H // 64), (H, I // 8), (H, I // 64), (H, I // 64)]
    dt = [np.uint32, np.uint16, np.uint16, np.uint32, np.uint16, np.uint16]
    names = ["gu_q", "gu_s", "gu_b", "d_q", "d_s", "d_b"]
    return {n: blob[o:o + sz].view(d).reshape(sh) for n, o, sz, sh, d in zip(names, off, sizes, shapes, dt)}


def test_untile_hand_worked_positions():
    g = _load("tile_layout.json")
    H, I = g["H"], g["I"]
    n = oracle.tile_blob_bytes(H, I)
    assert n == 24 * 576
    tiled = np.arange(n // 2, dtype=np.uint16).view(np.uint8)
    parts = _mlx_parts(oracle.untile_expert(tiled, H, I), H, I)
    words = tiled.view(np.uint32)
    for e in g["words"]:
        assert parts[e["part"]][e["row"], e["word"]] == words[e["tiled_word"]], e["why"]
    for e in g["halves"]:
        assert parts[e["part"]][e["row"], e["group"]] == e["tiled_half"], e["why"]


@pytest.mark.parametrize("H,I", [(128, 64), (256, 128), (384, 192)])
def test_untile_is_a_permutation(H, I):
    """Every halfword of the tile blob lands in exactly one MLX position and the
    sizes agree (no padding in either form at these shapes)."""
    n = oracle.tile_blob_bytes(H, I)
    assert n == oracle.expert_blob_bytes(H, I) == 3 * I * H * 36 // 64
    tiled = np.arange(n // 2, dtype=np.uint32).astype(np.uint16).view(np.uint8)
    if n // 2 > 65536:  # make halfwords unique with a second pass on the high part
        pytest.skip("shape too large for unique 16-bit tags")
    out = oracle.untile_expert(tiled, H, I).view(np.uint16)
    assert np.array_equal(np.sort(out), np.arange(n // 2, dtype=np.uint16))
