"""qerl_nvfp4_pack: the packed weight layout, byte for byte.

The layout is stated in include/qerl.h: one 18432-byte block per (128-row
tile t, 256-wide K stage g), blocks in (t, g) order; code bytes of row r at
r * 128 with 16-byte chunk c moved to chunk position c ^ (r % 8); scale pair p
(16-element blocks 2p, 2p+1) of row r at 16384 + 256 p + 2 r; zero padding.
Here that statement is written out with numpy index arithmetic and compared
with the kernel's output on random codes and scales, for shapes with ragged
row tiles and ragged K stages.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import nvfp4_weight_quantized_03_gb300 as mod
    mod.lib()
    return mod


def packed_reference(codes: np.ndarray, scales: np.ndarray, n: int, k: int) -> np.ndarray:
    tiles, stages = -(-n // 128), -(-k // 256)
    out = np.zeros((tiles, stages, 18432), dtype=np.uint8)
    for t in range(tiles):
        for g in range(stages):
            blk = out[t, g]
            for r in range(128):
                row = t * 128 + r
                if row >= n:
                    continue
                seg = codes[row, g * 128: g * 128 + 128]  # may be short in the last stage
                for c in range(len(seg) // 16):
                    pos = (c ^ (r % 8)) * 16
                    blk[r * 128 + pos: r * 128 + pos + 16] = seg[c * 16: c * 16 + 16]
                srow = scales[row, g * 16: g * 16 + 16]
                for p in range(len(srow) // 2):
                    blk[16384 + p * 256 + 2 * r: 16384 + p * 256 + 2 * r + 2] = srow[2 * p: 2 * p + 2]
    return out.reshape(-1)


@pytest.mark.parametrize("n,k", [(128, 256), (200, 320), (512, 3584), (17, 64), (384, 1088)])
def test_pack_matches_layout(q, n, k):
    rs = np.random.default_rng(n * 7919 + k)
    codes = rs.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    scales = rs.integers(0, 256, size=(n, k // 16), dtype=np.uint8)
    packed = q.pack(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda())
    assert packed.numel() == q.qerl_nvfp4_packed_size(n, k)
    assert np.array_equal(packed.cpu().numpy(), packed_reference(codes, scales, n, k))
