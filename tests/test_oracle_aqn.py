"""Pins for the oracle's AQN schedule and noise sampler.

QeRL digest, section 3.4 "Adaptive Quantization Noise (AQN)": Eq. 7
(Z ~ N(0, sigma^2 I), one value per input channel), Eq. 8 (exponential decay
sigma(k) = sigma_start (sigma_end / sigma_start)^((k-1)/(K-1)), k = 1..K) and
"Algorithm 1" (K stages of floor(M/K) steps).  Philox4x32-10 is from Salmon et
al., SC'11.
"""
import numpy as np
import pytest
from scipy import stats

from conftest import read_golden

G = {k: float(v) for k, v in read_golden("aqn_schedule.txt")}
S0, S1, K = G["sigma_start"], G["sigma_end"], int(G["num_stages"])


def test_philox_known_answers(orc):
    for row in read_golden("philox4x32_10_kat.txt"):
        vals = [int(h, 16) for h in row]
        out = orc.philox4x32_10(vals[0:4], vals[4:6])
        assert out.tolist() == vals[6:10]


def test_schedule_endpoints(orc):
    assert orc.aqn_sigma(0, K, S0, S1) == S0
    assert abs(orc.aqn_sigma(K - 1, K, S0, S1) - S1) <= 1e-15 * S1


def test_schedule_constant_ratio_and_symmetry(orc):
    sig = [orc.aqn_sigma(i, K, S0, S1) for i in range(K)]
    ratio = (S1 / S0) ** (1.0 / (K - 1))
    for a, b in zip(sig[:-1], sig[1:]):
        assert abs(b / a - ratio) <= 1e-14
        assert b < a
    # geometric interpolation: sigma(i) * sigma(K-1-i) = sigma_start * sigma_end
    for i in range(K):
        assert abs(sig[i] * sig[K - 1 - i] - S0 * S1) <= 1e-15 * S0 * S1 * 10


def test_schedule_special_stages(orc):
    assert orc.aqn_sigma(-1, K, S0, S1) == 0.0  # warm-up: quantization noise only
    assert orc.aqn_sigma(K + 5, K, S0, S1) == orc.aqn_sigma(K - 1, K, S0, S1)
    assert orc.aqn_sigma(0, 1, S0, S1) == S0 and orc.aqn_sigma(3, 1, S0, S1) == S0
    # Eq. 8 first drops below 2e-3 at its k = 6 (library stage 5)
    assert orc.aqn_sigma(4, K, S0, S1) > 2e-3 > orc.aqn_sigma(5, K, S0, S1)


def test_stage_mapping(orc):
    M = 8192
    per = M // K
    assert orc.aqn_stage(0, M, K) == 0
    assert orc.aqn_stage(per - 1, M, K) == 0
    assert orc.aqn_stage(per, M, K) == 1
    assert orc.aqn_stage(M - 1, M, K) == K - 1
    assert orc.aqn_stage(-3, M, K) == -1
    assert orc.aqn_stage(5, 3, K) == 5  # fewer steps than stages: one step per stage
    assert orc.aqn_stage(50, 3, K) == K - 1
    counts = np.bincount([orc.aqn_stage(s, 600, K) for s in range(600)])
    assert counts.tolist() == [60] * 10


def test_sampler_deterministic_and_streams_differ(orc):
    a = orc.aqn_sample(1003, 1.0, seed=7, stream_id=1, counter=5)
    b = orc.aqn_sample(1003, 1.0, seed=7, stream_id=1, counter=5)
    assert np.array_equal(a, b)
    for args in ((8, 1, 5), (7, 2, 5), (7, 1, 6)):
        c = orc.aqn_sample(1003, 1.0, seed=args[0], stream_id=args[1], counter=args[2])
        assert abs(np.corrcoef(a, c)[0, 1]) < 0.15
    # prefix property: channel j depends only on (j, seed, stream, counter)
    assert np.array_equal(orc.aqn_sample(13, 1.0, 7, 1, 5), a[:13])


def test_sampler_is_standard_normal_times_sigma(orc):
    n = 1_000_000
    z = orc.aqn_sample(n, 1.0, seed=123, stream_id=0, counter=0).astype(np.float64)
    assert abs(z.mean()) < 5 / np.sqrt(n)
    assert abs(z.std() - 1.0) < 5e-3
    assert stats.kstest(z, "norm").pvalue > 1e-4
    # 4-way interleave of the Box-Muller outputs: each lane is N(0,1) too
    for j in range(4):
        assert stats.kstest(z[j::4], "norm").pvalue > 1e-4
    assert abs(np.corrcoef(z[0::4], z[1::4])[0, 1]) < 5e-3


@pytest.mark.parametrize("sigma", [0.0, 5e-4, 1e-2, 3.0])
def test_sampler_scales_by_sigma(orc, sigma):
    s32 = float(np.float32(sigma))  # sigma is an fp32 argument
    z1 = orc.aqn_sample(4097, 1.0, 9, 0, 0).astype(np.float64)
    zs = orc.aqn_sample(4097, sigma, 9, 0, 0).astype(np.float64)
    # two fp32 roundings (of n and of sigma * n) separate the two sides
    assert np.all(np.abs(zs - s32 * z1) <= np.abs(s32 * z1) * 2 ** -23 + 1e-45)


# The digest's four decay schedules (AQN section, "Why exponential decay"; ablation Figures 9
# and 15): 0 exponential (Eq. 8), 1 linear, 2 cosine, 3 logarithmic.  Pinned by properties
# each closed form implies, not by retyping it.
SCHEDULES = (0, 1, 2, 3)


def _sched(orc, sch, k_stages=K):
    return [orc.aqn_sigma_schedule(sch, i, k_stages, S0, S1) for i in range(k_stages)]


def test_decay_schedules_share_stages_and_endpoints(orc):
    for sch in SCHEDULES:
        sig = _sched(orc, sch)
        assert sig[0] == S0
        assert abs(sig[-1] - S1) <= 1e-15 * S0
        assert all(b < a for a, b in zip(sig, sig[1:])), sch
        assert orc.aqn_sigma_schedule(sch, -1, K, S0, S1) == 0.0
        assert orc.aqn_sigma_schedule(sch, K + 3, K, S0, S1) == sig[-1]
        assert orc.aqn_sigma_schedule(sch, 2, 1, S0, S1) == S0
    assert np.isnan(orc.aqn_sigma_schedule(4, 1, K, S0, S1))
    assert np.isnan(orc.aqn_sigma_schedule(-1, 1, K, S0, S1))
    assert _sched(orc, 0) == [orc.aqn_sigma(i, K, S0, S1) for i in range(K)]


def test_linear_schedule_takes_equal_steps(orc):
    for k_stages in (2, 5, K):
        sig = _sched(orc, 1, k_stages)
        for a, b in zip(sig, sig[1:]):
            assert abs((a - b) - (S0 - S1) / (k_stages - 1)) <= 1e-17


def test_cosine_schedule_is_point_symmetric_and_s_shaped(orc):
    for k_stages in (9, K):
        sig = _sched(orc, 2, k_stages)
        for i in range(k_stages):
            assert abs(sig[i] + sig[k_stages - 1 - i] - (S0 + S1)) <= 1e-17
        if k_stages % 2:
            assert abs(sig[k_stages // 2] - (S0 + S1) / 2) <= 1e-17
        steps = [a - b for a, b in zip(sig, sig[1:])]
        mid = len(steps) // 2
        assert steps[0] < steps[mid] and steps[-1] < steps[mid]


def test_logarithmic_schedule_product_rule(orc):
    """The drop below sigma_start at stage k is proportional to log k: drop(k1 k2) = drop(k1) +
    drop(k2), and the drops per stage shrink (sharp start, long tail)."""
    def drop(k):
        return S0 - orc.aqn_sigma_schedule(3, k - 1, K, S0, S1)

    for k1, k2 in ((2, 2), (2, 3), (2, 4), (2, 5), (3, 3)):
        assert abs(drop(k1 * k2) - (drop(k1) + drop(k2))) <= 1e-17
    steps = [drop(k + 1) - drop(k) for k in range(1, K)]
    assert all(b < a for a, b in zip(steps, steps[1:]))
