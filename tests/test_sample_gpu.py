"""Token sampling (temperature, top-K, top-P, caller's uniform), CUDA path vs the
oracle, through the C ABI.

Logits are seeded N(0, 2^2) rows over vocabularies of 50 to 262,144 entries, with
planted exact ties (tied maximum, a block of equal values at the top-K boundary).
The GPU works in fp32 and the oracle in fp64, so a draw is compared only where no
decision (a top-P cut or the draw itself) lies within 1e-5 of its threshold,
relative to the kept total, as the oracle reports (the kernel's cumulative sums
carry about 1e-6 of relative error: an fp32 scan over at most 1024 weights).  With
a thousand kept tokens of tiny probability such near-ties occur; they are counted.
Exact ties are decided by index on both sides and are always compared.
"""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _rows(V, T, seed):
    rng = np.random.default_rng(seed)
    lg = (2.0 * rng.standard_normal((T, V))).astype(np.float32)
    if T > 1:
        lg[1, [3, V // 2, V - 1]] = lg[1].max() + 1.0       # tied maximum
    if T > 2 and V >= 100:
        top = np.sort(lg[2])[::-1]
        lg[2, rng.choice(V, 40, replace=False)] = top[30]    # a block of ties around rank 30
    u = rng.random(T).astype(np.float32)
    return lg, u


@pytest.mark.parametrize("V", [50, 1000, 32000, 262144])
def test_sample_matches_oracle(V):
    import bit_affine_quantised_affine4_b300 as moe
    T = 6
    compared = near = 0
    for seed, (temp, k, p) in enumerate([(0.2, 64, 0.95), (0.7, 8, 0.5), (1.5, 1024, 1.0), (0.0, 64, 0.95),
                                         (1.0, 1, 0.9), (0.9, 0 if V <= 1024 else 512, 0.99)]):
        lg, u = _rows(V, T, 100 * V + seed)
        tok = moe.moe_sample(torch.from_numpy(lg).cuda(), temp, k, p, torch.from_numpy(u).cuda())
        torch.cuda.synchronize()
        got = tok.cpu().numpy()
        for t in range(T):
            want, margin = oracle.sample(lg[t], temp, k, p, float(u[t]))
            if margin < 1e-5:
                near += 1
                continue
            compared += 1
            assert got[t] == want, (V, temp, k, p, t)
    assert compared >= 30 and near <= 6


def test_sample_exact_ties_and_greedy():
    import bit_affine_quantised_affine4_b300 as moe
    V, T = 5000, 4
    lg = np.zeros((T, V), np.float32)           # every logit equal: ties everywhere
    lg[1, 4000:] = 1.0                          # 1000 tied maxima
    u = np.array([0.0, 0.5, 0.999, 0.3], np.float32)
    for temp, k in ((0.0, 64), (1.0, 64), (0.5, 1000)):
        tok = moe.moe_sample(torch.from_numpy(lg).cuda(), temp, k, 1.0, torch.from_numpy(u).cuda())
        torch.cuda.synchronize()
        got = tok.cpu().numpy()
        for t in range(T):
            want, _ = oracle.sample(lg[t], temp, k, 1.0, float(u[t]))
            assert got[t] == want, (temp, k, t)


def test_sample_rejects_bad_arguments():
    import bit_affine_quantised_affine4_b300 as moe
    lg = torch.zeros((2, 5000), device="cuda")
    u = torch.zeros(2, device="cuda")
    for temp, k, p in ((1.0, 2000, 0.9), (1.0, 0, 0.9), (1.0, 64, 0.0), (1.0, 64, 1.5)):
        with pytest.raises(moe.MoeError) as e:
            moe.moe_sample(lg, temp, k, p, u)
        assert e.value.status == moe.MOE_EINVAL


def test_sample_large_vocab_both_paths():
    """262,144 logits: a row whose top bin holds 10,000 equal maxima (more than the
    4096 packs the compacting path keeps: the radix-select path runs) beside plain
    rows (the compacting path)."""
    import bit_affine_quantised_affine4_b300 as moe
    V, T = 262144, 3
    rng = np.random.default_rng(7)
    lg = (2.0 * rng.standard_normal((T, V))).astype(np.float32)
    lg[0, rng.choice(V, 10000, replace=False)] = lg[0].max() + 0.5
    u = rng.random(T).astype(np.float32)
    for temp, k, p in ((0.2, 64, 0.95), (1.0, 1000, 1.0)):
        tok = moe.moe_sample(torch.from_numpy(lg).cuda(), temp, k, p, torch.from_numpy(u).cuda())
        torch.cuda.synchronize()
        got = tok.cpu().numpy()
        for t in range(T):
            want, margin = oracle.sample(lg[t], temp, k, p, float(u[t]))
            if margin >= 1e-5:
                assert got[t] == want, (temp, k, p, t)
