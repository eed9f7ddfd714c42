"""The FMA-pipe 2^x used for part of the attention softmax, replayed on the
CPU in fp32 exactly as the kernel computes it (coefficients read from the
kernel header) and compared with numpy's exp2 (CPU)."""
import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "decoder_block_gb300", "csrc",
                   "ptx.cuh")


def _coeffs():
    text = open(HDR).read()
    c = {k: np.float32(float(v)) for k, v in re.findall(r"static constexpr float (kC\d) = ([0-9.eE+-]+)f;", text)}
    magic = np.float32(float(re.search(r"kMagic = ([0-9.]+)f;", text).group(1)))
    return c, magic


def _exp2_poly(x):
    c, magic = _coeffs()
    x = np.maximum(x.astype(np.float32), np.float32(-126.0))
    t = (x + magic).astype(np.float32)
    r = (t - magic).astype(np.float32)
    f = np.float32(-1.0) * r + x
    f = f.astype(np.float32)
    p = (c["kC3"] * f + c["kC2"]).astype(np.float32)
    p = (p * f + c["kC1"]).astype(np.float32)
    p = (p * f + c["kC0"]).astype(np.float32)
    n = (t.view(np.uint32) << np.uint32(23)).view(np.int32)
    return (p.view(np.int32) + n).view(np.float32)


def test_exp2_poly_relative_error_on_the_softmax_range():
    x = np.concatenate([np.linspace(-125.0, 8.0, 2_000_001, dtype=np.float32),
                        np.float32([-0.5, 0.5, 0.0, -1.0, 7.999, -0.4999, 0.4999])])
    y = _exp2_poly(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y - ref) / ref
    assert rel.max() < 1.0e-4  # the fit's 7.5e-5 plus fp32 evaluation; bf16 P needs 2^-9


def test_exp2_poly_underflow_and_minus_infinity():
    y = _exp2_poly(np.float32([-np.inf, -1000.0, -200.0, -126.0]))
    assert np.all(np.isfinite(y)) and np.all(y >= 0) and np.all(y < 2.0 ** -124)
