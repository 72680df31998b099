"""The v0.39.0 page's cache settings: defaults, the checks of its
configuration reference and troubleshooting list, and the byte accounting
of the defaults (host only)."""
import math

import numpy as np
import pytest

from query_aware_vq_gb300.config import A2ATSConfig


def test_defaults_are_the_pages():
    c = A2ATSConfig(head_dim=128).validate()
    assert (c.window, c.sub_dim, c.codebook_bits, c.use_query_aware) == (128, 8, 8, True)
    assert (c.beta, c.retrieval_fraction, c.b, c.rope_base) == (0.5, 0.20, 2048, 10000.0)
    assert c.n_centroids == 256


@pytest.mark.parametrize("kw,match", [
    (dict(head_dim=127), "even"),
    (dict(head_dim=0), "even"),
    (dict(head_dim=36), "multiple of sub_dim"),
    (dict(head_dim=128, beta=1.5), "beta"),
    (dict(head_dim=128, beta=math.nan), "beta"),
    (dict(head_dim=128, retrieval_fraction=-0.1), "retrieval_fraction"),
    (dict(head_dim=128, codebook_bits=0), "codebook_bits"),
    (dict(head_dim=128, query_h=np.eye(4)), "query_h"),
    (dict(head_dim=128, codebook=np.zeros((255, 8))), "codebook"),
    (dict(head_dim=128, rope_base=0.0), "rope_base"),
    (dict(head_dim=128, b=1 << 24), "b must"),
])
def test_rejected_settings(kw, match):
    with pytest.raises(ValueError, match=match):
        A2ATSConfig(**kw).validate()


def test_accepted_shapes():
    A2ATSConfig(head_dim=128, query_h=np.eye(8), codebook=np.zeros((256, 8))).validate()
    A2ATSConfig(head_dim=64, sub_dim=4, codebook_bits=4, query_h=np.zeros((8, 4, 4)),
                codebook=np.zeros((8, 16, 4))).validate()


def test_byte_accounting_of_the_defaults():
    from query_aware_vq_gb300 import build as qbuild
    qbuild.build()
    acc = A2ATSConfig(head_dim=128).byte_accounting(1000)
    assert acc["compression_ratio"] == 16.0
    assert acc["assigned_avg_bits"] == 1.0
    assert acc["codebook_bytes"] == 4096.0
    assert acc["compressed_key_bytes"] == acc["compressed_value_bytes"] == 1000 * 16
