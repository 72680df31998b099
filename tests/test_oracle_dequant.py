"""Pins of the oracle's dequantisation (v0.39.0 page, "How it works", step 3:
a key is reconstructed from its assigned centroid) and of the byte
accounting (v0.39.0 page, "Byte accounting" and "What you get with the
defaults"), the latter against the page's printed table."""
import numpy as np
import pytest

import oracle
from _golden import lines


def test_dequantize_is_the_centroid_of_each_code():
    rng = np.random.default_rng(0)
    K, d, n = 7, 5, 40
    c = rng.standard_normal((K, d))
    codes = rng.integers(0, K, n).astype(np.int32)
    codes[:3] = [-1, K, 1 << 30]
    out = oracle.dequantize(codes, c)
    assert (out[:3] == 0).all()
    np.testing.assert_array_equal(out[3:], c[codes[3:]])


def test_dequantize_inverts_an_exact_assignment():
    # keys that are centroids come back exactly from their own codes
    rng = np.random.default_rng(1)
    c = rng.standard_normal((16, 8))
    pick = rng.integers(0, 16, 100)
    code, _, _ = oracle.assign_cholesky(c[pick], c, None)
    np.testing.assert_array_equal(oracle.dequantize(code, c), c[pick])


@pytest.mark.parametrize("row", list(lines("compression_defaults.txt")))
def test_byte_accounting_matches_the_page_table(row):
    sub_dim, bits = int(row[0]), int(row[1])
    per_number, smaller, table_kb = float(row[2]), float(row[3]), float(row[4])
    acc = oracle.byte_accounting(tokens=1000, d=128, sub_dim=sub_dim, codebook_bits=bits)
    assert acc["assigned_avg_bits"] == per_number
    assert acc["compression_ratio"] == smaller
    assert acc["codebook_bytes"] / 1024 == table_kb
    assert acc["fp16_key_bytes"] == acc["fp16_value_bytes"] == 1000 * 128 * 2
    assert acc["compressed_key_bytes"] == acc["compressed_value_bytes"]
    # the stated bits per number times the numbers stored, in bytes
    assert acc["compressed_key_bytes"] == 1000 * 128 * per_number / 8


def test_byte_accounting_with_no_tokens_keeps_the_settings_ratio():
    acc = oracle.byte_accounting(tokens=0, d=128, sub_dim=8, codebook_bits=8)
    assert acc["compressed_key_bytes"] == acc["fp16_value_bytes"] == 0
    assert acc["compression_ratio"] == 16.0
