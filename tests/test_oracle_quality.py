"""The quality measurements of oracle.quality, pinned to textbook distortions and to the
logit-error relation Var(delta logit) = |q|^2 MSE / d ([turbo4 post-mortem] section 9)."""

import numpy as np
import pytest

from conftest import golden_lines
from oracle import quality


def max_distortion(levels):
    """Max's minimum mean-squared error for a unit Gaussian (the golden table's 2nd column)."""
    for ln in golden_lines("max_gaussian_quantizer.txt"):
        parts = ln.split()
        if int(parts[0]) == levels:
            return float(parts[1])
    raise KeyError(levels)


@pytest.mark.parametrize("label,args", quality.VARIANTS)
def test_logit_error_variance_is_mse_over_d(label, args):
    """Rotated-basis errors have no preferred direction, so the logit error variance over
    many (query, key) pairs matches |q|^2 MSE / d for every format and codebook."""
    mse, var, pred = quality.logit_error(quality.make_codec(args), n_keys=2048, n_queries=48, seed=3)
    assert abs(var - pred) / pred < 0.06


@pytest.mark.parametrize("fmt,levels", [("turbo4", 16), ("turbo3", 8)])
def test_lloyd_distortion_matches_max_table(fmt, levels):
    """Unit keys through the whole encode / dequantize path lose, per element and times d,
    what Max's table gives for the Gaussian Lloyd quantizer at that level count."""
    mse, _, _ = quality.logit_error(quality.make_codec(dict(fmt=fmt, codebook="lloyd")), n_keys=4096,
                                    n_queries=4, seed=5)
    assert abs(mse * quality.D / max_distortion(levels) - 1.0) < 0.03


def test_qjl_term_ablation_direction():
    """The unbiased QJL correction raises the key MSE above the 2-bit MSE stage alone (the
    ablation of [turbo4 post-mortem] section 3); the 2/pi-shrunk term lowers it."""
    args = dict(fmt="prod3", codebook="lloyd", qjl_seed=1001)
    full = quality.logit_error(quality.make_codec(args), n_keys=2048, n_queries=4, seed=7)[0]
    none = quality.logit_error(quality.make_codec(dict(args, drop_qjl=True)), n_keys=2048, n_queries=4, seed=7)[0]
    shrunk = quality.logit_error(quality.make_codec(dict(args, qjl_shrink=True)), n_keys=2048, n_queries=4,
                                 seed=7)[0]
    assert full > none > shrunk


def test_output_cosine_orders_formats():
    """16 Lloyd levels beat 8, which beat the 2-bit + QJL keys with 2-bit group values."""
    cos = {}
    for label, args in quality.VARIANTS:
        if label in ("turbo4 lloyd", "turbo3 lloyd", "prod3 lloyd"):
            kc = quality.make_codec(args)
            vc = (quality.Codec("vgroup2") if args["fmt"] == "prod3"
                  else quality.Codec(args["fmt"], rotation="dense", rot_seed=8, codebook="lloyd"))
            cos[label] = quality.output_cosine(kc, vc, L=1024, seed=9)[0]
    assert cos["turbo4 lloyd"] > cos["turbo3 lloyd"] > cos["prod3 lloyd"]
    assert cos["turbo4 lloyd"] > 0.97


@pytest.mark.parametrize("bits,levels", [(4, 16), (3, 8)])
def test_head_dim_256_halves_the_logit_noise(bits, levels):
    """[turbo4 post-mortem] section 9: with a codebook built for each head dimension, the
    per-element error times d is the same Gaussian distortion (Max's table), so the logit
    error variance |q|^2 MSE / d halves from d = 128 to d = 256."""
    r = {d: quality.head_dim_logit_error(d, bits, n_keys=2048, n_queries=48, seed=5) for d in (128, 256)}
    for d, (msed, var, pred) in r.items():
        assert abs(msed - max_distortion(levels)) / max_distortion(levels) < 0.03, d
        assert abs(var - pred) / pred < 0.06, d
    ratio = r[128][1] / r[256][1]
    assert 1.8 < ratio < 2.2
