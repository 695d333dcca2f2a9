"""GPU AQN sampler vs the oracle (Philox4x32-10 bits identical, Box-Muller in
fp64 on both sides, so z agrees to within one fp32 ulp)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import nvfp4_weight_quantized_03_gb300 as mod
    mod.lib()
    return mod


@pytest.mark.parametrize("k", [1, 3, 4, 5, 1000, 27648, (1 << 20) + 3])
@pytest.mark.parametrize("seed,stream_id,counter", [(0, 0, 0), (2**40 + 7, 3, 2**33 + 5)])
def test_sample_matches_oracle(q, orc, k, seed, stream_id, counter):
    z = torch.full((k,), 123.0, dtype=torch.float32, device="cuda")
    q.check(q.qerl_aqn_sample(z, 1e-2, seed, stream_id, counter))
    got = z.cpu().numpy()
    ref = orc.aqn_sample(k, 1e-2, seed, stream_id, counter)
    ulp = np.spacing(np.abs(ref).astype(np.float32))
    assert np.all(np.abs(got - ref) <= ulp), np.max(np.abs(got - ref) / ulp)


def test_sample_sigma_zero_and_schedule(q, orc):
    z = torch.full((100,), 1.0, dtype=torch.float32, device="cuda")
    q.check(q.qerl_aqn_sample(z, 0.0, 1, 0, 0))
    assert torch.count_nonzero(z).item() == 0
    for stage in range(10):
        sig = q.qerl_aqn_sigma(stage, 10, 1e-2, 5e-4)
        q.check(q.qerl_aqn_sample(z, sig, 5, 1, stage))
        ref = orc.aqn_sample(100, sig, 5, 1, stage)
        assert np.allclose(z.cpu().numpy(), ref, rtol=2 ** -22, atol=0)


def test_sample_statistics(q):
    z = torch.empty(1 << 22, dtype=torch.float32, device="cuda")
    q.check(q.qerl_aqn_sample(z, 2.0, 11, 0, 0))
    zz = z.double()
    assert abs(zz.mean().item()) < 5 * 2.0 / 2 ** 11
    assert abs(zz.std().item() - 2.0) < 5e-3
