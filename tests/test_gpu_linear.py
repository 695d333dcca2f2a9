"""GPU NVFP4 + LoRA + AQN linear vs the fp64 oracle.

Bound (fp32 accumulation, bf16 output): normwise ||y - bf16(y_hat)|| / ||y_hat||
<= 1e-3 and max |y - bf16(y_hat)| / max |y_hat| <= 2e-3, with y_hat the oracle's
fp64 result on the same seeded inputs.  Small shapes are compared in full and
span several 128-row tiles, several 64-wide K stages and ragged M / N tails;
the workload shapes are compared on sampled output columns (and rows).
"""
import numpy as np
import pytest
import torch

import workloads as wl
from helpers import assert_linear_close, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import nvfp4_weight_quantized_03_gb300 as mod
    mod.lib()
    return mod


_QCACHE = {}


def _quantized(q, orc, n, k, seed):
    key = (n, k, seed)
    if key not in _QCACHE:
        if len(_QCACHE) > 4:
            _QCACHE.clear()
        W = wl.weight_f32(n, k, seed, 0)
        codes, scales, S = q.quantize(torch.from_numpy(W).cuda())
        oc, osc, oS = orc.quantize(W)
        assert np.array_equal(codes.cpu().numpy(), oc)
        assert np.array_equal(scales.cpu().numpy(), osc)
        assert S.item() == float(oS)
        _QCACHE[key] = (q.pack(codes, scales), S, oc, osc, oS)
    return _QCACHE[key]


class Case:
    """One seeded problem: weights quantized on the GPU (checked bit-exact
    against the oracle), inputs shared by both sides."""

    def __init__(self, q, orc, m, n, k, r, sigma, seed=0, x_std=1.0):
        self.m, self.n, self.k, self.r = m, n, k, r
        self.x_bits = wl.activations_bits(m, k, seed, 1, std=x_std)
        self.A_bits = wl.lora_A_bits(r, k, seed, 2) if r else None
        self.B_bits = wl.lora_B_bits(n, r, seed, 3) if r else None
        self.z = wl.noise_vector(k, sigma, seed, 4) if sigma else None
        self.alpha = 2.0 * r
        self.wp, self.S, self.oc, self.osc, self.oS = _quantized(q, orc, n, k, seed)
        self.x = dev_bf16(self.x_bits)
        self.A = dev_bf16(self.A_bits) if r else None
        self.B = dev_bf16(self.B_bits) if r else None
        self.zd = torch.from_numpy(self.z).cuda() if sigma else None

    def gpu(self, q, out_dtype=torch.bfloat16, ws=None):
        y = torch.full((self.m, self.n), float("nan"), dtype=out_dtype, device="cuda")
        ws = ws if ws is not None else q.workspace(q.qerl_lora_linear_workspace_size(self.m, self.n, self.k, self.r))
        q.check(q.qerl_lora_linear(self.x, self.wp, self.S, self.zd, self.A, self.B, self.alpha, y, ws))
        assert q.qerl_read_status(ws) == 0
        return y

    def oracle(self, orc, rows=None, cols=None):
        xb = self.x_bits if rows is None else self.x_bits[rows]
        return orc.lora_linear(xb, self.oc, self.osc, self.oS, z=self.z, A_bits=self.A_bits, B_bits=self.B_bits,
                               alpha=self.alpha, cols=cols)


SMALL = [
    # m, n, k, r, sigma
    (1, 128, 64, 0, 0.0),
    (4, 2048, 2048, 16, 1e-2),  # the 3B q_proj single-linear workload, in full
    (3, 200, 320, 8, 1e-2),
    (16, 256, 1024, 32, 5e-3),
    (17, 384, 1024, 32, 5e-3),
    (100, 130, 512, 16, 1e-2),
    (128, 512, 2048, 32, 1e-2),
    (129, 256, 512, 16, 1e-2),
    (256, 256, 256, 32, 1e-2),
    (300, 300, 576, 32, 1e-2),
    (600, 256, 256, 128, 1e-2),
    (8, 512, 3584, 32, 1e-2),  # 7B k/v shape at decode (K split across a cluster)
    (32, 1024, 4096, 16, 0.0),
    # 65..128 tokens, single tiles (pair mode needs >= 12 weight stages per CTA)
    (100, 384, 2048, 128, 1e-2),  # rank 128 (late LoRA operand)
    (72, 1000, 1024, 32, 1e-2),   # ragged N
    (128, 256, 6144, 32, 1e-2),   # K split across a cluster
    (65, 128, 512, 8, 0.0),       # one tile
    (48, 384, 3584, 128, 1e-2),   # rank 128 at 33..64 tokens: the LoRA operand built late, in the idle ring
    (128, 512, 18944, 128, 5e-3), # rank 128 at 128 tokens, long K (summed LoRA groups)
    # 33..64 tokens
    (40, 512, 2048, 32, 1e-2),
    (64, 768, 3584, 16, 5e-3),
    # several 128-token tiles (> 128 tokens)
    (257, 512, 2048, 32, 1e-2),   # 3 token tiles, ragged last rows
    (384, 256, 1536, 16, 5e-3),
    (512, 1024, 2048, 0, 1e-2),   # 4 token tiles, no LoRA
    (300, 256, 2048, 128, 1e-2),  # rank 128
    # pair mode (two 128-row tiles per CTA sharing the activation slabs; >= 12 weight stages)
    (257, 512, 3072, 32, 1e-2),   # 12 stages, 3 token tiles, ragged last rows
    (130, 384, 4096, 16, 5e-3),   # 16 stages, 2 token tiles; the second pair has one tile
]


@pytest.mark.parametrize("m,n,k,r,sigma", SMALL)
def test_linear_small_full(q, orc, m, n, k, r, sigma):
    c = Case(q, orc, m, n, k, r, sigma)
    y = c.gpu(q)
    assert_linear_close(y, c.oracle(orc), orc, what=f"m{m} n{n} k{k} r{r}")


def test_linear_fp32_output(q, orc):
    c = Case(q, orc, 5, 384, 512, 16, 1e-2)
    y = c.gpu(q, torch.float32)
    norm, mx = assert_linear_close(y, c.oracle(orc), orc, bf16_out=False)
    assert norm < 1e-5 and mx < 1e-5  # fp32 output: only accumulation order differs


def test_linear_zero_noise_equals_no_noise(q, orc):
    c = Case(q, orc, 6, 256, 512, 16, 1e-2)
    c.zd = torch.zeros_like(c.zd)
    a = c.gpu(q, torch.float32)
    c.zd = None
    b = c.gpu(q, torch.float32)
    # the LoRA reduction order may differ between calls; the base part is identical
    assert torch.allclose(a, b, rtol=1e-6, atol=1e-7)


def test_linear_extreme_activation_scales(q, orc):
    for std in (1e-20, 1e4):
        c = Case(q, orc, 4, 256, 512, 16, 1e-2, seed=3, x_std=std)
        assert_linear_close(c.gpu(q), c.oracle(orc), orc, what=f"x_std {std}")


def test_linear_workspace_reuse_and_status(q, orc):
    c1 = Case(q, orc, 8, 384, 1024, 32, 1e-2, seed=1)
    c2 = Case(q, orc, 64, 256, 512, 16, 1e-2, seed=2)
    ws = q.workspace(max(q.qerl_lora_linear_workspace_size(8, 384, 1024, 32),
                         q.qerl_lora_linear_workspace_size(64, 256, 512, 16)))
    for _ in range(2):
        assert_linear_close(c1.gpu(q, ws=ws), c1.oracle(orc), orc)
        assert_linear_close(c2.gpu(q, ws=ws), c2.oracle(orc), orc)


def test_linear_empty(q):
    ws = q.workspace(256)
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    wp = torch.zeros(q.qerl_nvfp4_packed_size(128, 64), dtype=torch.uint8, device="cuda")
    S = torch.ones(1, device="cuda")
    y = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    assert q.qerl_lora_linear(x, wp, S, None, None, None, 0.0, y, ws) == 0


def _sample_cols(n, cnt, seed):
    rs = np.random.default_rng(seed)
    cols = np.unique(np.concatenate([[0, n - 1], rs.choice(n, cnt, replace=False)]))
    return cols


@pytest.mark.parametrize("m", [1, 8, 32, 128])
@pytest.mark.parametrize("lin", wl.QWEN_7B, ids=lambda l: l.name)
def test_linear_7b_decode_sampled(q, orc, m, lin):
    """Qwen2.5-7B decoder-layer linears at decode batch m, r=32, alpha=64."""
    c = Case(q, orc, m, lin.n, lin.k, 32, 1e-2, seed=7)
    c.alpha = 64.0
    y = c.gpu(q)
    cols = _sample_cols(lin.n, 48, m)
    assert_linear_close(y[:, torch.from_numpy(cols).cuda()], c.oracle(orc, cols=cols), orc,
                        what=f"7B {lin.name} m{m}")


@pytest.mark.parametrize("lin", [wl.QWEN_14B[0], wl.QWEN_14B[6]], ids=lambda l: l.name)
def test_linear_14b_prefill_sampled(q, orc, lin):
    """Qwen2.5-14B linears at prefill M=4096, r=32, alpha=64, sigma=5e-3; sampled rows x columns."""
    m = 4096
    c = Case(q, orc, m, lin.n, lin.k, 32, 5e-3, seed=14)
    c.alpha = 64.0
    y = c.gpu(q)
    rows = _sample_cols(m, 24, 1)
    cols = _sample_cols(lin.n, 24, 2)
    sub = y[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()]
    assert_linear_close(sub, c.oracle(orc, rows=rows, cols=cols), orc, what=f"14B {lin.name} prefill")


@pytest.mark.parametrize("m", [1, 8, 128])
def test_linear_group_matches_single_calls(q, orc, m):
    """q/k/v-like group (three linears of one input, different N, ranks and alphas, one without
    LoRA): every output matches its own qerl_lora_linear call and the oracle."""
    k = 1024
    shapes = [(768, 16, 32.0), (256, 8, 24.0), (384, 0, 0.0)]
    cases = [Case(q, orc, m, n, k, r, 1e-2, seed=40 + i) for i, (n, r, _) in enumerate(shapes)]
    x = cases[0].x
    for c, (_, _, alpha) in zip(cases, shapes):
        c.x, c.x_bits, c.z, c.zd = x, cases[0].x_bits, cases[0].z, cases[0].zd
        c.alpha = alpha
    ys = [torch.full((m, c.n), float("nan"), dtype=torch.bfloat16, device="cuda") for c in cases]
    lin = [(c.wp, c.S, c.A, c.B, c.alpha, y) for c, y in zip(cases, ys)]
    ws = q.workspace(q.qerl_lora_linear_group_workspace_size(m, k, lin))
    q.check(q.qerl_lora_linear_group(x, cases[0].zd, lin, ws))
    assert q.qerl_read_status(ws) == 0
    for c, y in zip(cases, ys):
        assert_linear_close(y, c.oracle(orc), orc, what=f"group n{c.n} r{c.r}")
        single = c.gpu(q)
        assert torch.allclose(y.float(), single.float(), rtol=1e-2, atol=1e-3)
    # the same group through a descriptor array built once: the same launch, bit for bit
    ys2 = [torch.full_like(y, float("nan")) for y in ys]
    arr = q.linear_descs([(c.wp, c.S, c.A, c.B, c.alpha, y) for c, y in zip(cases, ys2)])
    for _ in range(2):
        q.check(q.qerl_lora_linear_group(x, cases[0].zd, arr, ws))
    assert q.qerl_read_status(ws) == 0
    for y, y2 in zip(ys, ys2):
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_linear_group_four_with_an_empty_member(q, orc):
    m, k = 8, 512
    cases = [Case(q, orc, m, n, k, 16, 0.0, seed=50 + i) for i, n in enumerate([256, 128, 512])]
    x = cases[0].x
    for c in cases:
        c.x, c.x_bits = x, cases[0].x_bits
    ys = [torch.full((m, c.n), float("nan"), dtype=torch.bfloat16, device="cuda") for c in cases]
    empty_y = torch.empty((m, 0), dtype=torch.bfloat16, device="cuda")
    lin = [(c.wp, c.S, c.A, c.B, c.alpha, y) for c, y in zip(cases, ys)]
    lin.insert(1, (cases[0].wp, cases[0].S, None, None, 0.0, empty_y))
    ws = q.workspace(q.qerl_lora_linear_group_workspace_size(m, k, lin))
    q.check(q.qerl_lora_linear_group(x, None, lin, ws))
    assert q.qerl_read_status(ws) == 0
    for c, y in zip(cases, ys):
        assert_linear_close(y, c.oracle(orc), orc, what=f"group4 n{c.n}")


def test_linear_full_wave_separate_activation_ring(q, orc):
    """100 tokens (separate activation ring) over 152 tiles of 128 rows: one CTA per tile,
    no K split, a full wave.  Full output against the oracle."""
    c = Case(q, orc, 100, 152 * 128, 512, 16, 1e-2, seed=31)
    assert_linear_close(c.gpu(q), c.oracle(orc), orc, what="full wave")


def test_linear_group_full_wave_two_members(q, orc):
    """A grouped launch of 75 + 77 tiles at 96 tokens (ragged last tile): the members' tiles
    are consecutive on the grid, no K split."""
    m, k = 96, 512
    cases = [Case(q, orc, m, n, k, 16, 1e-2, seed=60 + i) for i, n in enumerate([75 * 128, 77 * 128 - 40])]
    x = cases[0].x
    for c in cases:
        c.x, c.x_bits, c.z, c.zd = x, cases[0].x_bits, cases[0].z, cases[0].zd
    ys = [torch.full((m, c.n), float("nan"), dtype=torch.bfloat16, device="cuda") for c in cases]
    lin = [(c.wp, c.S, c.A, c.B, c.alpha, y) for c, y in zip(cases, ys)]
    ws = q.workspace(q.qerl_lora_linear_group_workspace_size(m, k, lin))
    q.check(q.qerl_lora_linear_group(x, cases[0].zd, lin, ws))
    assert q.qerl_read_status(ws) == 0
    for c, y in zip(cases, ys):
        assert_linear_close(y, c.oracle(orc), orc, what=f"wave group n{c.n}")


GUARD = 4096
GUARD_BYTE = 0xA5


def _guarded(nbytes):
    """A device byte buffer of nbytes followed by GUARD bytes of a pattern."""
    buf = torch.full((nbytes + GUARD,), GUARD_BYTE, dtype=torch.uint8, device="cuda")
    return buf


def _guard_intact(buf, nbytes):
    return bool((buf[nbytes:] == GUARD_BYTE).all().item())


@pytest.mark.parametrize("m,n,k,r", [(8, 384, 1024, 32), (100, 384, 2048, 32), (300, 256, 576, 16)])
def test_no_writes_past_the_buffers(q, orc, m, n, k, r):
    """Guard regions after y, the workspace and the packed weights stay untouched by the
    quantizer, the packer and the linear (decode, pair and prefill paths; ragged N)."""
    W = wl.weight_f32(n, k, 91, 0)
    codes, scales, S = q.quantize(torch.from_numpy(W).cuda())
    pbytes = q.qerl_nvfp4_packed_size(n, k)
    pbuf = _guarded(pbytes)
    q.check(q.qerl_nvfp4_pack(codes, scales, pbuf[:pbytes]))
    torch.cuda.synchronize()
    assert _guard_intact(pbuf, pbytes), "pack wrote past the packed weights"
    x = dev_bf16(wl.activations_bits(m, k, 92, 1))
    A, B = dev_bf16(wl.lora_A_bits(r, k, 93, 2)), dev_bf16(wl.lora_B_bits(n, r, 94, 3))
    zd = torch.from_numpy(wl.noise_vector(k, 1e-2, 95)).cuda()
    wsb = q.qerl_lora_linear_workspace_size(m, n, k, r)
    wsb = (wsb + 255) // 256 * 256
    wbuf = _guarded(wsb)
    wbuf[:wsb].zero_()
    ybytes = m * n * 2
    ybuf = _guarded(ybytes)
    y = ybuf[:ybytes].view(torch.bfloat16).view(m, n)
    for _ in range(2):
        q.check(q.qerl_lora_linear(x, pbuf[:pbytes], S, zd, A, B, 2.0 * r, y, wbuf[:wsb]))
    assert q.qerl_read_status(wbuf[:wsb]) == 0
    assert _guard_intact(ybuf, ybytes), "the linear wrote past y"
    assert _guard_intact(wbuf, wsb), "the linear wrote past its workspace"
    assert _guard_intact(pbuf, pbytes), "the linear wrote into the packed weights' guard"
    rows = None if m <= 128 else np.arange(0, m, 9)
    ref = orc.lora_linear(wl.activations_bits(m, k, 92, 1) if rows is None else wl.activations_bits(m, k, 92, 1)[rows],
                          *orc.quantize(W), z=wl.noise_vector(k, 1e-2, 95), A_bits=wl.lora_A_bits(r, k, 93, 2),
                          B_bits=wl.lora_B_bits(n, r, 94, 3), alpha=2.0 * r)
    assert_linear_close(y if rows is None else y[torch.from_numpy(rows).cuda()], ref, orc, what="guarded")


def test_linear_group_pair_mode_several_token_tiles(q, orc):
    """A grouped launch at 260 tokens (3 token tiles, pair mode: 12 weight stages) of two members
    with different tile counts and ranks."""
    m, k = 260, 3072
    cases = [Case(q, orc, m, n, k, r, 1e-2, seed=90 + i) for i, (n, r) in enumerate([(512, 32), (768, 16)])]
    x = cases[0].x
    for c in cases:
        c.x, c.x_bits, c.z, c.zd = x, cases[0].x_bits, cases[0].z, cases[0].zd
    ys = [torch.full((m, c.n), float("nan"), dtype=torch.bfloat16, device="cuda") for c in cases]
    lin = [(c.wp, c.S, c.A, c.B, c.alpha, y) for c, y in zip(cases, ys)]
    ws = q.workspace(q.qerl_lora_linear_group_workspace_size(m, k, lin))
    q.check(q.qerl_lora_linear_group(x, cases[0].zd, lin, ws))
    assert q.qerl_read_status(ws) == 0
    for c, y in zip(cases, ys):
        assert_linear_close(y, c.oracle(orc), orc, what=f"pair group m{m} n{c.n}")
