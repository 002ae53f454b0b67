"""The input generators' FP8 storage formats against the oracle's independent
decoders: what a row stores is what the oracle reads back, within E4M3's
rounding (3 mantissa bits: a relative half-step of 2^-4 for normal values)."""
import numpy as np
import torch

import oracle
from long_context_sparse_26_b300 import workloads as wl


def _f64(t):
    return oracle.bf16_bits_to_f64(t.contiguous().view(torch.int16).numpy().view(np.uint16))


def test_fp8_latent_rows_decode_to_their_source():
    kv = wl.latent_cache(2, 40, 11, 0, "cpu")
    kv[0, 3, 128:256] = 0                                   # an all-zero group
    rows = wl.to_fp8_latent(kv)
    assert rows.dtype == torch.uint8 and tuple(rows.shape) == (2, 40, oracle.FP8_LATENT_ROW_BYTES)
    got = oracle.fp8_latent_to_f64(rows.numpy())
    want = _f64(kv)
    assert np.array_equal(got[..., 512:], want[..., 512:])  # RoPE dims stored as they are
    assert not got[0, 3, 128:256].any()
    nope_w, nope_g = want[..., :512].reshape(2, 40, 4, 128), got[..., :512].reshape(2, 40, 4, 128)
    amax = np.abs(nope_w).max(axis=-1, keepdims=True)
    scale = np.where(amax > 0, amax / 448.0, 1.0)
    # each value within half an E4M3 step of its scaled source (subnormal steps are 2^-9 x scale)
    step = np.maximum(np.abs(nope_w) * 2.0 ** -3, 2.0 ** -9 * scale)
    assert np.all(np.abs(nope_g - nope_w) <= 0.5 * step + 1e-12)
    # the group maximum is represented exactly (it maps to the largest code)
    idx = np.abs(nope_w).argmax(axis=-1)
    gmax = np.take_along_axis(nope_g, idx[..., None], -1)
    wmax = np.take_along_axis(nope_w, idx[..., None], -1)
    nz = wmax != 0
    assert np.allclose(gmax[nz], wmax[nz], rtol=1e-6, atol=0)


def test_e4m3_rows_decode_to_their_source():
    k = wl.indexer_keys(2, 50, 13, "cpu")
    codes, scale = wl.to_e4m3_rows(k)
    assert codes.dtype == torch.uint8 and tuple(codes.shape) == (2, 50, 128) and tuple(scale.shape) == (2, 50)
    got = oracle.e4m3_to_f64(codes.numpy()) * scale.double().numpy()[..., None]
    want = _f64(k)
    sc = scale.double().numpy()[..., None]
    step = np.maximum(np.abs(want) * 2.0 ** -3, 2.0 ** -9 * sc)
    assert np.all(np.abs(got - want) <= 0.5 * step + 1e-12)
