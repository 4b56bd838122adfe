"""GPU quantisers against the oracle's codecs, bit for bit: MXFP8 blocks of 32
(E8M0 scale + E4M3 elements) and FP8 latent rows (fp32 scale per row or per
128-dim tile + E4M3 latent dims, bf16 rope dims), over N(0,1) data and the edge cases (all-zero blocks,
tiny and huge magnitudes, blocks whose E8M0 scale clamps at 2^-127, exact
ties to even)."""
import numpy as np
import pytest
import torch

from _util import dev_bf16
from indexer_top_sparse_gb300.inputs import bf16_bits

pytestmark = pytest.mark.gpu


def _data(rng, shape):
    x = rng.standard_normal(shape).astype(np.float32)
    flat = x.reshape(-1, x.shape[-1])
    flat[0, :32] = 0.0
    flat[1, :32] *= np.float32(1e-30)
    flat[2, 32:64] *= np.float32(1e30)
    flat[3, :32] = np.float32(1.0625) * np.float32(2.0) ** rng.integers(-20, 20, 32).astype(np.float32)
    # blocks whose scale clamps to the smallest E8M0 byte (amax below 2^-119:
    # bf16 subnormals and the smallest normals), and one near the bf16 maximum
    flat[4, :32] *= np.float32(2.0 ** -130)
    flat[4, 32:64] *= np.float32(2.0 ** -124)
    flat[5, :32] *= np.float32(2.0 ** -121)
    flat[5, 32:64] = np.float32(3.38e38) * np.sign(flat[5, 32:64])
    return x


def test_mxfp8_bit_exact(orc):
    rng = np.random.default_rng(0)
    bits = bf16_bits(_data(rng, (37, 64, 128)))
    import indexer_top_sparse_gb300 as d
    q, e = d.dsa_quant_mxfp8(dev_bf16(bits))
    rq, re = orc.quant_mxfp8(bits)
    assert np.array_equal(e.cpu().numpy(), re)
    assert np.array_equal(q.cpu().numpy(), rq)


def test_fp8_rows_bit_exact(orc):
    rng = np.random.default_rng(1)
    x = _data(rng, (300, 576))
    x[7, :512] = 0.0
    x[8] *= np.float32(1e-3)
    bits = bf16_bits(x)
    import indexer_top_sparse_gb300 as d
    nope, rope, sc = d.dsa_quant_fp8_rows(dev_bf16(bits))
    rn, rr, rs = orc.quant_fp8_rows(bits)
    assert np.array_equal(sc.cpu().numpy(), rs)
    assert np.array_equal(nope.cpu().numpy(), rn)
    assert np.array_equal(rope.view(torch.int16).cpu().numpy().view(np.uint16), rr)


def test_fp8_tiles_bit_exact(orc):
    # one scale per 128 latent dims: all-zero tiles next to live ones, tiles of
    # very different magnitude in one row, a ragged row count
    rng = np.random.default_rng(2)
    x = _data(rng, (301, 576))
    x[7, :512] = 0.0
    x[9, 128:256] = 0.0
    x[10, 384:512] *= np.float32(1e20)
    x[11, 256:384] *= np.float32(1e-20)
    bits = bf16_bits(x)
    import indexer_top_sparse_gb300 as d
    nope, rope, sc = d.dsa_quant_fp8_tiles(dev_bf16(bits))
    rn, rr, rs = orc.quant_fp8_tiles(bits)
    assert tuple(sc.shape) == (301, 4)
    assert np.array_equal(sc.cpu().numpy(), rs)
    assert np.array_equal(nope.cpu().numpy(), rn)
    assert np.array_equal(rope.view(torch.int16).cpu().numpy().view(np.uint16), rr)
