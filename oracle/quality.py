"""Quality of the compressed formats on synthetic data (oracle; test infrastructure only).

[turbo4 post-mortem] section 9 explains format quality through the logit error: with
attention logits q.k / sqrt(d), a key error e whose coordinates have variance MSE (per
element) and no preferred direction gives Var(delta logit) = |q|^2 MSE / d, so at a fixed
per-element MSE a head dimension of 128 has twice the logit noise of 256, and going from
8 to 16 centroids cuts the MSE and hence the noise.  This module measures both sides of
that argument for every (format, codebook) the library offers, and the end effect on
attention outputs (cosine against exact fp64 attention over the uncompressed K and V,
the quality side-metric of the method's write-ups).

Run ``python -m oracle.quality`` for the tables (the second compares head dimensions
64, 128 and 256 with a codebook built for each).  Inputs are seeded synthetic draws
(``synth``); no dataset is used.
"""

import math

import numpy as np

from .attention import attention_reference
from .formats import Codec

D = 128

# (label, key codec arguments) of every rotated key format and codebook
VARIANTS = [
    ("turbo4 quantile", dict(fmt="turbo4", codebook="quantile")),
    ("turbo4 lloyd", dict(fmt="turbo4", codebook="lloyd")),
    ("turbo4 sphere", dict(fmt="turbo4", codebook="sphere")),
    ("turbo3 lloyd", dict(fmt="turbo3", codebook="lloyd")),
    ("turbo3 sphere", dict(fmt="turbo3", codebook="sphere")),
    ("prod3 lloyd", dict(fmt="prod3", codebook="lloyd", qjl_seed=1001)),
    ("prod3 lloyd, QJL x 2/pi", dict(fmt="prod3", codebook="lloyd", qjl_seed=1001, qjl_shrink=True)),
    ("prod3 lloyd, no QJL term", dict(fmt="prod3", codebook="lloyd", qjl_seed=1001, drop_qjl=True)),
]


def make_codec(args, rotation="dense", rot_seed=7):
    args = dict(args)
    drop = args.pop("drop_qjl", False)
    codec = Codec(rotation=rotation, rot_seed=rot_seed, **args)
    if drop:
        codec.qjl_factor = 0.0
    return codec


def logit_error(codec, n_keys=4096, n_queries=64, seed=0):
    """Per-element key MSE and the variance of the logit error over all (query, key) pairs.

    Keys are unit vectors (N(0,1) rows normalised), queries N(0,1) rows; the logit is
    q.k / sqrt(d).  Returns (mse_per_element, var_logit_error, predicted = E|q|^2 mse / d).
    """
    rng = np.random.default_rng([seed, 11])
    k = rng.standard_normal((n_keys, D))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = rng.standard_normal((n_queries, D))
    blocks, _ = codec.encode(k.astype(np.float32))
    e = codec.dequantize(blocks) - k.astype(np.float32).astype(np.float64)
    mse = float(np.mean(e * e))
    dl = (q @ e.T) / math.sqrt(D)
    return mse, float(np.var(dl)), float(np.mean(np.sum(q * q, axis=1)) * mse / D)


def output_cosine(kcodec, vcodec, L=2048, Hq=4, seed=0, lognormal=True):
    """Cosine of the attention output over compressed K and V against exact fp64 attention
    over the uncompressed ones: one KV head, Hq query heads, L keys drawn like the GQA
    workload (lognormal channel scales with one outlier channel) when lognormal.
    Returns (mean, min) over the query heads."""
    rng = np.random.default_rng([seed, 12])
    scale = np.exp(rng.normal(0.0, 0.5, D)) if lognormal else np.ones(D)
    if lognormal:
        scale[rng.integers(D)] *= 8.0
    k = (rng.standard_normal((L, D)) * scale).astype(np.float32)
    v = (rng.standard_normal((L, D)) * scale).astype(np.float32)
    q = rng.standard_normal((1, Hq, D))
    exact, _ = attention_reference(q, k[None, None].astype(np.float64), v[None, None].astype(np.float64))
    kh = kcodec.dequantize(kcodec.encode(k)[0])[None, None]
    vh = vcodec.dequantize(vcodec.encode(v)[0])[None, None]
    approx, _ = attention_reference(q, kh, vh)
    cos = np.sum(exact * approx, axis=-1) / (np.linalg.norm(exact, axis=-1) * np.linalg.norm(approx, axis=-1))
    return float(cos.mean()), float(cos.min())


def head_dim_logit_error(d, bits=4, kind="lloyd", n_keys=4096, n_queries=64, seed=0):
    """Logit error of a d-dimensional head quantized as one block: a seeded dense rotation
    of the whole head (QR of a Gaussian matrix), nearest-centroid coding of every rotated
    coordinate with the codebook built for dimension d (the "per-head-dim codebook" of
    [turbo4 post-mortem] section 9), the norm kept exactly.  Keys are unit vectors,
    queries N(0, 1) rows, logits q.k / sqrt(d).  Returns (mse_per_element * d,
    var_logit_error, predicted = E|q|^2 mse / d).

    This is a study of the quality argument at other head dimensions; the packed formats
    and the GPU path are defined for d = 128."""
    from .codebook import make_codebook, stored_codebook

    rng = np.random.default_rng([seed, 13, d])
    rot, rr = np.linalg.qr(rng.standard_normal((d, d)))
    rot = rot * np.sign(np.diag(rr))  # unique orthogonal factor (diag(R) > 0)
    c32, b32 = stored_codebook(make_codebook(bits, d, kind))
    k = rng.standard_normal((n_keys, d))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = rng.standard_normal((n_queries, d))
    y = k @ rot.T
    idx = np.sum(y[:, :, None] > b32.astype(np.float64)[None, None, :], axis=2)
    k_hat = c32.astype(np.float64)[idx] @ rot
    e = k_hat - k
    mse = float(np.mean(e * e))
    dl = (q @ e.T) / math.sqrt(d)
    return mse * d, float(np.var(dl)), float(np.mean(np.sum(q * q, axis=1)) * mse / d)


def report(seed=0):
    """Rows of (label, MSE x d, Var(delta logit), predicted, cosine mean, cosine min); values
    use the same format for K and V except prod3 keys, which pair with vgroup2 values."""
    rows = []
    for label, args in VARIANTS:
        kc = make_codec(args)
        mse, var, pred = logit_error(kc, seed=seed)
        if args["fmt"] == "prod3":
            vc = Codec("vgroup2")
        else:
            vc = Codec(args["fmt"], rotation="dense", rot_seed=8, codebook=args["codebook"])
        cmean, cmin = output_cosine(kc, vc, seed=seed)
        rows.append((label, mse * D, var, pred, cmean, cmin))
    return rows


def main():
    print("| keys (values) | MSE x d | Var(delta logit) | |q|^2 MSE / d | output cosine mean | min |")
    print("|---|---|---|---|---|---|")
    for label, msed, var, pred, cmean, cmin in report():
        vals = "vgroup2" if label.startswith("prod3") else label.split()[0] + " " + label.split()[1]
        print(f"| {label} ({vals}) | {msed:.5f} | {var:.3e} | {pred:.3e} | {cmean:.6f} | {cmin:.6f} |")
    print()
    print("| head dim | bits | MSE x d | Var(delta logit) | |q|^2 MSE / d |")
    print("|---|---|---|---|---|")
    for d in (64, 128, 256):
        for bits in (4, 3):
            msed, var, pred = head_dim_logit_error(d, bits)
            print(f"| {d} | {bits} | {msed:.5f} | {var:.3e} | {pred:.3e} |")


if __name__ == "__main__":
    main()
