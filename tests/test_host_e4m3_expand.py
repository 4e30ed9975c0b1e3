"""The bit map the MXFP8 converter warps use to expand E4M3 codes to bf16,
restated in numpy and checked against the oracle's E4M3 table on every code
(OCP 8-bit floating point spec, E4M3: bias 7, subnormals 0.mmm x 2^-6, no
infinities, NaN at S.1111.111, which the quantizer never writes).

The map must give the bf16 bits of 2^-120 times the code's value:
`prmt.b32` with selector nibbles whose bit 3 is set replicates the selected
byte's sign bit over the result byte (PTX ISA, prmt default mode), so each
code lands in a 16-bit lane as a signed v, and (v & 0x087f) << 4 is the
result. The multiply-add map an earlier converter used,
16 * (c + 15 * (c & 0x80)) for a code byte c in a 16-bit lane, is checked
too, as a second derivation of the same bits.
The scale multiply that follows (bf16, by 2^(e + 120)) is exact while the
product stays normal; that step is checked on the GPU against the oracle."""
from __future__ import annotations

import numpy as np

import oracle


def prmt(a: np.ndarray, b: int, sel: int) -> np.ndarray:
    """prmt.b32 d, a, b, sel in the default mode, on uint32 arrays."""
    src = [(a >> np.uint32(8 * i)) & np.uint32(0xFF) for i in range(4)]
    src += [np.full_like(a, (b >> (8 * i)) & 0xFF) for i in range(4)]
    out = np.zeros_like(a)
    for i in range(4):
        n = (sel >> (4 * i)) & 0xF
        byte = src[n & 7]
        if n & 8:
            byte = np.where(byte & np.uint32(0x80), np.uint32(0xFF), np.uint32(0))
        out |= byte << np.uint32(8 * i)
    return out


def bf16_value(bits16: np.ndarray) -> np.ndarray:
    return (bits16.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def codes_words():
    """Every non-NaN code in every byte position of a 32-bit word."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint32)
    rng = np.random.default_rng(7)
    words = []
    for pos in range(4):
        others = rng.choice(codes, size=(codes.size, 4))
        others[:, pos] = codes
        words.append(others[:, 0] | others[:, 1] << 8 | others[:, 2] << 16 | others[:, 3] << 24)
    return np.concatenate(words).astype(np.uint32)


def expected(words: np.ndarray, byte: int) -> np.ndarray:
    table = oracle.e4m3_values().astype(np.float64)
    return table[(words >> np.uint32(8 * byte)) & np.uint32(0xFF)] * 2.0 ** -120


def test_multiply_add_route_matches_e4m3_table():
    w = codes_words()
    for sel, pair in ((0x4140, (0, 1)), (0x4342, (2, 3))):
        a = prmt(w, 0, sel)
        r = ((a + np.uint32(15) * (a & np.uint32(0x00800080))) << np.uint32(4)).astype(np.uint32)
        for h, byte in enumerate(pair):
            got = bf16_value((r >> np.uint32(16 * h)) & np.uint32(0xFFFF))
            assert np.array_equal(got, expected(w, byte)), (hex(sel), byte)


def test_sign_extending_permute_route_matches_e4m3_table():
    w = codes_words()
    for sel, pair in ((0x9180, (0, 1)), (0xB3A2, (2, 3))):
        v = prmt(w, 0, sel)
        r = ((v & np.uint32(0x087F087F)) << np.uint32(4)).astype(np.uint32)
        for h, byte in enumerate(pair):
            got = bf16_value((r >> np.uint32(16 * h)) & np.uint32(0xFFFF))
            assert np.array_equal(got, expected(w, byte)), (hex(sel), byte)


def test_permute_sign_replication_reading():
    # selector nibble 8 | i: the sign of byte i over the whole result byte
    a = np.array([0x00_80_7F_01], dtype=np.uint32)
    assert prmt(a, 0, 0x9180)[0] == 0x0000_0001 | 0x007F_0000
    assert prmt(np.array([0x0000_8081], dtype=np.uint32), 0, 0x9180)[0] == 0xFF80_FF81
