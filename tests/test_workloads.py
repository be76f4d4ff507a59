"""The seeded generators give matrices with the character each configuration
states (sparsity, mean row length, row-length CoV): the statistics the
pages use to tell deep-learning matrices from scientific ones ("Sparse GPU
Kernels for Deep Learning", "Interesting ideas" I1-I2).  CPU only."""
import math

import pytest

import workloads as W


def binomial_cov(n, p):
    return math.sqrt((1 - p) / (n * p))


def test_tiny():
    st = W.stats(W.tiny().csr)
    assert abs(st["sparsity"] - 0.90) < 0.01
    assert st["row_length_cov"] == pytest.approx(binomial_cov(256, 0.1), rel=0.2)


def test_resnet():
    st = W.stats(W.resnet(with_sddmm=False).csr)
    assert abs(st["sparsity"] - 0.80) < 0.005
    assert st["row_length_cov"] == pytest.approx(binomial_cov(2048, 0.2), rel=0.15)   # ~0.05


@pytest.mark.parametrize("shape", W.FFN_SHAPES, ids=["4096x1024", "1024x4096"])
@pytest.mark.parametrize("s", W.FFN_SPARSITIES)
def test_ffn(shape, s):
    M, K = shape
    st = W.stats(W.ffn(M, K, s, with_spmm=False, with_sddmm=False).csr)
    assert abs(st["sparsity"] - s / 100) < 0.005
    assert abs(st["row_length_cov"] - 0.1) < 0.01


@pytest.mark.parametrize("s", W.LSTM_SPARSITIES)
def test_lstm(s):
    st = W.stats(W.lstm(s).csr)
    assert abs(st["sparsity"] - s / 100) < 0.005
    assert st["row_length_cov"] == pytest.approx(binomial_cov(4096, 1 - s / 100), rel=0.15)


def test_attention():
    p = W.attention()
    st = W.stats(p.csr)
    assert abs(st["mean_row_length"] - 410) < 5          # ~90% sparsity within a head's 4096 keys
    assert abs(st["row_length_cov"] - 0.5) < 0.03        # lognormal, clipped to [1, 4096]
    assert p.csr.seg_rows == 4096 and p.csr.M == 8 * 4096
