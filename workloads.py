"""Seeded synthetic inputs for the NVFP4 + LoRA + AQN linear.

This module only draws random numbers in the shapes and distributions of the
workloads; it contains none of the method's arithmetic (no quantization, no
noise application, no linear algebra).  Both the CUDA path and the oracle are
fed from here, and nothing here depends on either of them.

Every tensor comes from its own numpy PCG64 stream derived from
(seed, *path), e.g. (0, layer, projection, role), so any single tensor can be
regenerated without drawing the others.  bf16 tensors are returned as uint16
bit patterns (round-to-nearest-even from the fp32 draw, done by torch).

Workload shapes are the Qwen2.5 linears used by QeRL's experiments
("QeRL: Beyond Efficiency", section 5 "Experiments"; shapes given as
N x K = out x in features).
"""
from dataclasses import dataclass

import numpy as np
import torch

# ---- shapes ---------------------------------------------------------------


@dataclass(frozen=True)
class Linear:
    name: str
    n: int  # output features
    k: int  # input features
    group: str  # AQN noise group: qkv, o, gate_up, down


def decoder_layer(hidden: int, inter: int, kv: int):
    """The seven LoRA-carrying linears of one decoder block, N x K."""
    return [
        Linear("q", hidden, hidden, "qkv"),
        Linear("k", kv, hidden, "qkv"),
        Linear("v", kv, hidden, "qkv"),
        Linear("o", hidden, hidden, "o"),
        Linear("gate", inter, hidden, "gate_up"),
        Linear("up", inter, hidden, "gate_up"),
        Linear("down", hidden, inter, "down"),
    ]


QWEN_3B_QPROJ = Linear("q", 2048, 2048, "qkv")
QWEN_7B = decoder_layer(3584, 18944, 512)
QWEN_14B = decoder_layer(5120, 13824, 1024)
QWEN_32B = decoder_layer(5120, 27648, 1024)
QWEN_7B_LAYERS = 28
QWEN_32B_LAYERS = 64

NOISE_GROUPS = ("qkv", "o", "gate_up", "down")

# ---- random streams ---------------------------------------------------------


def rng(seed: int, *path: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), *[int(p) for p in path]])))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), nearest-even, via torch."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---- tensors ----------------------------------------------------------------


def outlier_channels(k: int, seed: int, *path: int, frac: float = 0.005) -> np.ndarray:
    """Indices of the input channels (columns of W) that carry outliers:
    round(frac * k) of them, chosen by a seeded permutation."""
    cnt = int(round(frac * k))
    return np.sort(rng(seed, *path, 7).permutation(k)[:cnt])


def weight_f32(n: int, k: int, seed: int, *path: int, std: float = 0.02, outlier_frac: float = 0.005,
               outlier_scale: float = 10.0) -> np.ndarray:
    """W [n, k] fp32 ~ N(0, std^2) with round(outlier_frac * k) input channels scaled by outlier_scale."""
    W = rng(seed, *path, 1).standard_normal((n, k), dtype=np.float32) * np.float32(std)
    cols = outlier_channels(k, seed, *path, frac=outlier_frac)
    W[:, cols] *= np.float32(outlier_scale)
    return W


def weight_heavy_tail_bf16(n: int, k: int, seed: int, *path: int, std: float = 0.02, outlier_frac: float = 0.005,
                           nu: float = 3.0) -> np.ndarray:
    """bf16 bits [n, k]: N(0, std^2) with round(outlier_frac * k) input channels drawn
    from std * Student-t(nu) instead (heavy-tailed outlier channels)."""
    g = rng(seed, *path, 2)
    W = g.standard_normal((n, k), dtype=np.float32) * np.float32(std)
    cols = outlier_channels(k, seed, *path, frac=outlier_frac)
    W[:, cols] = (g.standard_t(nu, size=(n, cols.size)) * std).astype(np.float32)
    return to_bf16_bits(W)


def activations_bits(m: int, k: int, seed: int, *path: int, std: float = 1.0) -> np.ndarray:
    """x [m, k] bf16 bits ~ N(0, std^2)."""
    return to_bf16_bits(rng(seed, *path, 3).standard_normal((m, k), dtype=np.float32) * np.float32(std))


def lora_A_bits(r: int, k: int, seed: int, *path: int) -> np.ndarray:
    """A [r, k] bf16 bits ~ N(0, 1/k) (LoRA down-projection, r x in_features)."""
    return to_bf16_bits(rng(seed, *path, 4).standard_normal((r, k), dtype=np.float32) * np.float32(1.0 / np.sqrt(k)))


def lora_B_bits(n: int, r: int, seed: int, *path: int, std: float = 0.01) -> np.ndarray:
    """B [n, r] bf16 bits ~ N(0, std^2) (LoRA up-projection, out_features x r)."""
    return to_bf16_bits(rng(seed, *path, 5).standard_normal((n, r), dtype=np.float32) * np.float32(std))


def rmsnorm_weight_bits(k: int, seed: int, *path: int, mean: float = 1.0, std: float = 0.1) -> np.ndarray:
    """An RMSNorm scale w [k] bf16 bits ~ |N(mean, std^2)| (positive, around 1, as trained
    norm scales are; synthetic)."""
    return to_bf16_bits(np.abs(rng(seed, *path, 8).standard_normal(k, dtype=np.float32) * np.float32(std)
                               + np.float32(mean)))


def noise_vector(k: int, sigma: float, seed: int, *path: int) -> np.ndarray:
    """A channel-wise noise vector z [k] fp32 = sigma * N(0, 1), drawn on the host.
    (Used as a plain input of the linear; the library's own sampler is separate.)"""
    return (rng(seed, *path, 6).standard_normal(k) * sigma).astype(np.float32)


# ---- device-side draws for the large benchmark workloads ---------------------


def torch_generator(seed: int, *path: int, device="cuda") -> torch.Generator:
    """A torch generator on `device` seeded from (seed, *path) via SeedSequence."""
    s = int(np.random.SeedSequence([int(seed), *[int(p) for p in path]]).generate_state(1, dtype=np.uint64)[0])
    g = torch.Generator(device=device)
    g.manual_seed(s & ((1 << 63) - 1))
    return g


def weight_f32_device(n: int, k: int, seed: int, *path: int, std: float = 0.02, outlier_frac: float = 0.005,
                      outlier_scale: float = 10.0, device="cuda") -> torch.Tensor:
    """Device fp32 W [n, k] ~ N(0, std^2) with round(outlier_frac * k) input channels x outlier_scale."""
    g = torch_generator(seed, *path, 1, device=device)
    W = torch.randn((n, k), generator=g, device=device, dtype=torch.float32) * std
    cols = torch.from_numpy(outlier_channels(k, seed, *path, frac=outlier_frac)).to(device)
    W[:, cols] *= outlier_scale
    return W


def weight_heavy_tail_bf16_device(n: int, k: int, seed: int, *path: int, std: float = 0.02,
                                  outlier_frac: float = 0.005, nu: int = 3, device="cuda") -> torch.Tensor:
    """Device bf16 W [n, k] ~ N(0, std^2), with round(outlier_frac * k) input channels drawn
    from std * Student-t(nu) instead (t = Z / sqrt(chi2_nu / nu), chi2_nu a sum of nu squared
    normals; integer nu)."""
    g = torch_generator(seed, *path, 2, device=device)
    W = torch.randn((n, k), generator=g, device=device, dtype=torch.float32) * std
    cols = torch.from_numpy(outlier_channels(k, seed, *path, frac=outlier_frac)).to(device)
    z = torch.randn((n, cols.numel()), generator=g, device=device, dtype=torch.float32)
    chi2 = torch.zeros_like(z)
    for _ in range(nu):
        chi2 += torch.randn(z.shape, generator=g, device=device, dtype=torch.float32) ** 2
    W[:, cols] = z / torch.sqrt(chi2 / nu) * std
    return W.to(torch.bfloat16)


def normal_bf16_device(shape, std: float, seed: int, *path: int, device="cuda") -> torch.Tensor:
    g = torch_generator(seed, *path, 3, device=device)
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)
