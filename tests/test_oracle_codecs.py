"""Pins for the oracle's scalar codecs and quantisers, against the OCP format
tables, torch's own float8 dtypes (a library decoder/encoder) and brute-force
nearest-code search."""
import json
import math
import os

import numpy as np
import pytest
import torch

from indexer_top_sparse_gb300.inputs import bf16_bits, bf16_to_f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ocp_fp8_points.json")


def _torch_e4m3_decode_all():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def test_e4m3_spec_points(orc):
    g = json.load(open(GOLDEN))
    for code, val in g["e4m3"]:
        got = orc.e4m3_to_f64(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), code


def test_e8m0_spec_points(orc):
    g = json.load(open(GOLDEN))
    for code, val in g["e8m0"]:
        got = orc.e8m0_to_f64(int(code, 16))
        assert (math.isnan(got) if val == "nan" else got == val), code


def test_e4m3_decode_matches_torch_all_codes(orc):
    ref = _torch_e4m3_decode_all()
    for c in range(256):
        got = orc.e4m3_to_f64(c)
        if math.isnan(ref[c]):
            assert math.isnan(got)
        else:
            assert got == ref[c], hex(c)


def test_e8m0_decode_matches_torch(orc):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    for c in range(256):
        got = orc.e8m0_to_f64(c)
        assert (math.isnan(got) and math.isnan(ref[c])) or got == ref[c], c


def test_bf16_decode_matches_torch(orc):
    bits = np.arange(0, 65536, 37, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    for b, r in zip(bits, ref):
        got = orc.bf16_to_f64(int(b))
        assert (math.isnan(got) and math.isnan(r)) or got == r


def _nearest_e4m3_bruteforce(x, table):
    """Nearest finite E4M3 code to x, ties to the even code (mantissa LSB 0),
    by exhaustive search; saturates at +-448."""
    finite = [c for c in range(256) if not math.isnan(table[c])]
    best = None
    for c in finite:
        d = abs(table[c] - x)
        key = (d, c & 1)
        # prefer sign-matching zero
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_e4m3_encode_is_nearest_even_bruteforce(orc):
    table = _torch_e4m3_decode_all()
    rng = np.random.default_rng(1)
    xs = list(rng.standard_normal(400) * 30) + list(rng.standard_normal(200) * 0.01)
    # exact midpoints between neighbouring positive codes, and the codes themselves
    pos = sorted({table[c] for c in range(0x00, 0x7F)})
    xs += [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])] + pos
    for x in xs:
        c = orc.f64_to_e4m3(x)
        want = _nearest_e4m3_bruteforce(x, table)
        assert table[c] == table[want], (x, hex(c), hex(want))
        if table[c] == 0.0:
            continue
        assert (c & 1) == (want & 1), (x, hex(c), hex(want))


def test_e4m3_encode_matches_torch_in_range(orc):
    rng = np.random.default_rng(2)
    xs = np.concatenate([rng.standard_normal(3000) * 40, rng.standard_normal(1000) * 1e-3]).astype(np.float32)
    xs = xs[np.abs(xs) <= 448]
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.f64_to_e4m3(float(x)) for x in xs], np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates(orc):
    for x in [448.0, 449.0, 470.0, 480.0, 1e9, float("inf")]:
        assert orc.f64_to_e4m3(x) == 0x7E
        assert orc.f64_to_e4m3(-x) == 0xFE


def test_e4m3_roundtrip_all_finite_codes(orc):
    for c in range(256):
        v = orc.e4m3_to_f64(c)
        if math.isnan(v):
            continue
        assert orc.f64_to_e4m3(v) == c


def test_mxfp8_quant_properties(orc):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((6, 128)).astype(np.float32) * np.float32(3.0)
    x[0, :32] = 0.0                         # all-zero block
    x[1, :32] *= np.float32(1e-20)          # tiny block
    x[2, 32:64] *= np.float32(1e15)         # huge block
    bits = bf16_bits(x)
    xv = bf16_to_f32(bits).astype(np.float64)
    q, e = orc.quant_mxfp8(bits)
    assert q.shape == (6, 128) and e.shape == (6, 4)
    table = _torch_e4m3_decode_all()
    for r in range(6):
        for g in range(4):
            blk = xv[r, g * 32:(g + 1) * 32]
            amax = np.abs(blk).max()
            if amax == 0:
                assert e[r, g] == 127 and np.all(q[r, g * 32:(g + 1) * 32] == 0)
                continue
            sc = 2.0 ** (int(e[r, g]) - 127)
            # the scale is the power of two that puts amax in [256, 512)
            assert 256.0 <= amax / sc < 512.0
            for i in range(32):
                c = int(q[r, g * 32 + i])
                want = _nearest_e4m3_bruteforce(min(max(blk[i] / sc, -448.0), 448.0), table)
                assert table[c] == table[want]
            deq = np.array([table[c] for c in q[r, g * 32:(g + 1) * 32]]) * sc
            sat = np.abs(blk / sc) > 448.0
            assert np.all(np.abs(deq[sat]) == 448.0 * sc)
            normal = (np.abs(blk) >= 2.0 ** -6 * sc) & ~sat
            assert np.all(np.abs(deq - blk)[normal] <= 2.0 ** -4 * np.abs(blk)[normal])


def test_mxfp8_scale_clamps_to_the_e8m0_range(orc):
    # OCP MX v1.0: the block scale is 2^X with X = floor(log2 amax) - 8 (the
    # E4M3 emax), stored as the E8M0 byte X + 127, whose range is 2^-127 ..
    # 2^127.  A block with amax below 2^-119 (the smallest bf16 normals and the
    # bf16 subnormals) would need X < -127: the byte clamps to 0 and the
    # elements are x / 2^-127 rounded to the nearest E4M3 (no saturation is
    # possible there, |x| / 2^-127 < 2^8).  The largest finite bf16 magnitude
    # (2 - 2^-7) 2^127 gives X = 119, byte 246, so bf16 input never reaches the
    # upper end of the range.
    rng = np.random.default_rng(31)
    exps = [-133, -132, -131, -130, -129, -128, -127, -126, -125, -121, -120, -119, -118, -100]
    x = np.zeros((len(exps) + 1, 32), np.float32)
    for i, e in enumerate(exps):
        x[i] = (rng.random(32).astype(np.float32) + np.float32(0.5)) * np.float32(2.0 ** e)
        x[i, ::3] *= np.float32(-1.0)
    bits = bf16_bits(x)
    bits[-1] = np.where(np.arange(32) % 2 == 0, 0x7F7F, 0xFF00).astype(np.uint16)  # +max bf16, -2^127
    xv = bf16_to_f32(bits).astype(np.float64)
    q, e = orc.quant_mxfp8(bits)
    table = _torch_e4m3_decode_all()
    clamped = 0
    for r in range(x.shape[0]):
        amax = np.abs(xv[r]).max()
        assert amax > 0.0
        X = math.frexp(amax)[1] - 1 - 8            # floor(log2 amax) - 8, exact
        want_byte = min(max(X + 127, 0), 254)
        clamped += want_byte != X + 127
        assert int(e[r, 0]) == want_byte, (r, amax, X)
        sc = 2.0 ** (want_byte - 127)
        for i in range(32):
            want = _nearest_e4m3_bruteforce(min(max(xv[r, i] / sc, -448.0), 448.0), table)
            assert table[int(q[r, i])] == table[want], (r, i)
    assert int(e[-1, 0]) == 246
    assert clamped >= 8    # the clamped blocks are really exercised


def test_fp8_row_quant_matches_library_cast(orc):
    rng = np.random.default_rng(4)
    kv = rng.standard_normal((9, 576)).astype(np.float32)
    kv[3, :512] = 0.0
    kv[4] *= np.float32(1e-3)
    bits = bf16_bits(kv)
    nope, rope, scale = orc.quant_fp8_rows(bits)
    assert np.array_equal(rope, bits[:, 512:])
    xv = bf16_to_f32(bits)
    for r in range(9):
        amax = np.float32(np.abs(xv[r, :512]).max())
        s = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(448.0))
        assert scale[r] == s
        y = (xv[r, :512] / s).astype(np.float32)
        y = np.clip(y, -448.0, 448.0).astype(np.float32)
        ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(nope[r], ref), r


def test_fp8_tile_quant_matches_library_cast(orc):
    # one scale per 128 latent dims: tiles of very different magnitude, an
    # all-zero tile (scale 1) and an all-zero row
    rng = np.random.default_rng(5)
    kv = rng.standard_normal((7, 576)).astype(np.float32)
    kv[1, 128:256] = 0.0
    kv[2, :512] = 0.0
    kv[3, 256:384] *= np.float32(1e-3)
    kv[4, 384:512] *= np.float32(300.0)
    bits = bf16_bits(kv)
    nope, rope, scale = orc.quant_fp8_tiles(bits)
    assert scale.shape == (7, 4)
    assert np.array_equal(rope, bits[:, 512:])
    xv = bf16_to_f32(bits)
    for r in range(7):
        for j in range(4):
            tile = xv[r, 128 * j:128 * (j + 1)]
            amax = np.float32(np.abs(tile).max())
            s = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(448.0))
            assert scale[r, j] == s, (r, j)
            y = np.clip((tile / s).astype(np.float32), -448.0, 448.0).astype(np.float32)
            ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(nope[r, 128 * j:128 * (j + 1)], ref), (r, j)


def test_fp8_tile_quant_equals_row_quant_when_tiles_share_amax(orc):
    # with the same amax in all four tiles the tile scales all equal the row
    # scale, so the two quantisers must produce the same codes
    rng = np.random.default_rng(6)
    kv = rng.standard_normal((5, 576)).astype(np.float32)
    for j in range(4):
        kv[:, 128 * j + 7] = np.float32(9.5)
    bits = bf16_bits(kv)
    n_t, r_t, s_t = orc.quant_fp8_tiles(bits)
    n_r, r_r, s_r = orc.quant_fp8_rows(bits)
    assert np.array_equal(n_t, n_r) and np.array_equal(r_t, r_r)
    assert np.array_equal(s_t, np.repeat(s_r[:, None], 4, axis=1))
