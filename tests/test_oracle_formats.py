"""Pins for the oracle's decoders and dequantisers (CPU only).

Each check ties the oracle to something other than itself: a library's own
decoder (numpy float16, torch bfloat16 / float8_e4m3fn), closed forms from the
format definitions, hand-worked blocks, and the record sizes the pages print.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth


def test_fp16_all_codes_match_numpy():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode("fp16", codes)
    ref = codes.view(np.float16).astype(np.float64)
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(ours[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


def test_bf16_all_codes_match_torch():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode("bf16", codes)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(ours[m], ref[m])


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode("e4m3", codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(ours[m], ref[m])


def test_e4m3_definition_points():
    # OCP 8-bit floating point spec, E4M3: bias 7, max normal 448 (S.1111.110),
    # min normal 2^-6, min subnormal 2^-9, only S.1111.111 is NaN.
    d = lambda c: float(oracle.decode("e4m3", np.array([c], dtype=np.uint8))[0])
    assert d(0x00) == 0.0 and math.copysign(1, d(0x80)) == -1
    assert d(0x01) == 2.0 ** -9
    assert d(0x07) == 7 * 2.0 ** -9
    assert d(0x08) == 2.0 ** -6
    assert d(0x38) == 1.0 and d(0xB8) == -1.0
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0
    assert d(0x78) == 256.0
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))


def test_e2m1_all_codes_closed_form():
    # OCP FP4 E2M1: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 for codes 0..7,
    # bit 3 is the sign.
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    ours = oracle.decode("e2m1", np.arange(16, dtype=np.uint8))
    for c in range(16):
        want = mags[c & 7] * (-1.0 if c & 8 else 1.0)
        assert ours[c] == want, c
    assert math.copysign(1, ours[8]) == -1.0


def _q4_block(d_bits, qbytes):
    return np.concatenate([np.array([d_bits & 0xFF, d_bits >> 8], dtype=np.uint8),
                           np.asarray(qbytes, dtype=np.uint8)])


def test_q4_0_hand_worked_blocks():
    # Block layout: fp16 scale d, then 16 bytes; byte i holds element i (low
    # nibble) and element i+16 (high nibble); w = d * (q - 8).
    blocks = []
    expect = []
    # codes all 8 -> zeros
    blocks.append(_q4_block(0x3C00, [0x88] * 16)); expect.append([0.0] * 32)
    # codes all 0, d = 1 -> -8
    blocks.append(_q4_block(0x3C00, [0x00] * 16)); expect.append([-8.0] * 32)
    # d = 0.5, low nibble i, high nibble 15-i
    blocks.append(_q4_block(0x3800, [i | ((15 - i) << 4) for i in range(16)]))
    expect.append([0.5 * (i - 8) for i in range(16)] + [0.5 * (7 - i) for i in range(16)])
    # d = -2, low 0, high 15
    blocks.append(_q4_block(0xC000, [0xF0] * 16)); expect.append([16.0] * 16 + [-14.0] * 16)
    # subnormal scale 2^-24, low 15, high 9
    blocks.append(_q4_block(0x0001, [0x9F] * 16)); expect.append([7 * 2.0 ** -24] * 16 + [2.0 ** -24] * 16)
    mat = np.concatenate(blocks)
    got = oracle.dequant_matrix("q4_0", mat, rows=len(blocks), cols=32)
    assert np.array_equal(got, np.array(expect))
    # two blocks per row keep their order along the row
    got2 = oracle.dequant_matrix("q4_0", mat[: 4 * 18], rows=2, cols=64)
    assert np.array_equal(got2[0], np.array(expect[0] + expect[1]))
    assert np.array_equal(got2[1], np.array(expect[2] + expect[3]))


def test_fp8_tile_scales_index_rows_then_cols():
    rows, cols = 256, 384  # 2 x 3 tiles of 128 x 128
    q = np.full(rows * cols, 0x38, dtype=np.uint8)  # every code is 1.0
    scales = np.array([1, 2, 3, 5, 7, 11], dtype=np.float32)  # row-major over the tile grid
    mat = np.concatenate([q, scales.view(np.uint8)])
    w = oracle.dequant_matrix("fp8_b128", mat, rows, cols)
    for bi in range(2):
        for bj in range(3):
            tile = w[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            assert np.all(tile == scales[bi * 3 + bj])
    # ragged edge: 130 x 200 -> 2 x 2 tiles, last tile partial
    rows, cols = 130, 200
    q = np.full(rows * cols, 0xB0, dtype=np.uint8)  # -0.5
    sc = np.array([1, 2, 4, 8], dtype=np.float32)
    w = oracle.dequant_matrix("fp8_b128", np.concatenate([q, sc.view(np.uint8)]), rows, cols)
    assert w[129, 199] == -0.5 * 8 and w[0, 128] == -0.5 * 2 and w[128, 0] == -0.5 * 4


def test_nvfp4_hand_block():
    # one row of 32 weights = 2 blocks of 16; codes 0..15 in order (low nibble
    # = even element), block scales e4m3 0x38 (1.0) and 0x40 (2.0), g = 0.25
    codes = np.array([(2 * i) | ((2 * i + 1) << 4) for i in range(8)] * 2, dtype=np.uint8)
    mat = np.concatenate([codes, np.array([0x38, 0x40], dtype=np.uint8)])
    w = oracle.dequant_matrix("nvfp4", mat, rows=1, cols=32, g=0.25)
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    e2m1 = [mags[c & 7] * (-1.0 if c & 8 else 1.0) for c in range(16)]
    want = [v * 1.0 * 0.25 for v in e2m1] + [v * 2.0 * 0.25 for v in e2m1]
    assert np.array_equal(w[0], np.array(want))


def test_q4_0_matches_numpy_float16_bulk():
    # bulk check of the block walk against numpy's float16 decoder on random bytes
    rng = np.random.default_rng(5)
    rows, cols = 7, 96
    nb = cols // 32
    mat = rng.integers(0, 256, size=rows * nb * 18, dtype=np.uint8)
    blk = mat.reshape(rows, nb, 18)
    d = blk[:, :, :2].copy().view(np.float16)[..., 0].astype(np.float64)
    q = blk[:, :, 2:]
    ok = np.isfinite(d)
    lo = (q & 15).astype(np.float64) - 8
    hi = (q >> 4).astype(np.float64) - 8
    ref = (np.concatenate([lo, hi], axis=2) * d[..., None]).reshape(rows, cols)
    got = oracle.dequant_matrix("q4_0", mat, rows, cols)
    fin = np.repeat(ok, 32, axis=1)
    assert np.array_equal(got[fin], ref[fin])


def test_record_sizes_against_pages():
    # Q4_0 at the explainer's expert shape (3 matrices of 2560 x 640): the
    # NVMe build's contiguous 2,764,800-byte blocks, "2.64 MiB" per expert.
    assert oracle.slot_bytes("q4_0", 2560, 640) == 2764800
    assert round(2764800 / 2 ** 20, 2) == 2.64
    # Qwen3-30B-A3B shape (H 2048, I 768)
    assert oracle.slot_bytes("q4_0", 2048, 768) == 2654208
    assert oracle.slot_bytes("fp8_b128", 2048, 768) == 4719744
    # the dev.to page: ~4.72 MB per FP8 expert with scales ignored; x 48 layers ~ 227 MB per slot
    assert round(3 * 2048 * 768 / 1e6, 2) == 4.72
    assert round(48 * 4719744 / 1e6) == 227
    assert oracle.slot_bytes("nvfp4", 2048, 768) == 2654208
    assert oracle.record_bytes("nvfp4", 2048, 768) == 2654208 + 12
    assert oracle.slot_bytes("bf16", 256, 128) == 196608
    # synth lays records out with the same geometry
    for f in ("bf16", "q4_0", "fp8_b128", "nvfp4"):
        assert synth.record_bytes(f, 2048, 768) == oracle.record_bytes(f, 2048, 768)


@pytest.mark.parametrize("fmt", ["bf16", "q4_0", "fp8_b128", "nvfp4"])
def test_synth_records_decode_finite(fmt):
    H, I = 256, 128
    rec = synth.expert_record(fmt, 7, 0, 3, H, I)
    mb = oracle.matrix_bytes(fmt, I, H)
    w = oracle.dequant_matrix(fmt, rec[:mb], I, H, g=1.0)
    assert np.all(np.isfinite(w))
    assert w.std() > 0
    # regenerating the same expert gives the same bytes; another expert differs
    assert np.array_equal(rec, synth.expert_record(fmt, 7, 0, 3, H, I))
    assert not np.array_equal(rec, synth.expert_record(fmt, 7, 0, 4, H, I))
    many = synth.expert_records(fmt, 7, 0, 2, 3, H, I)
    assert np.array_equal(many[1], rec)
