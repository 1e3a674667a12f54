"""Calibrates the per-layer Zipf popularity bias of the skewed decode stack.

The dev.to page ("A hot expert cache made a 181 GiB model faster", section
"Offload more, cache the hot experts") reports that within one layer the
hottest 35% of the experts take 74% of the picks.  The synthetic stack gets
that skew from a bias b_e = -alpha * ln(rank_e) added to the router logits.
An unbiased router with W_r ~ N(0, 0.05^2) and x ~ N(0, 1) gives, per token,
logits that are close to iid N(0, (0.05 sqrt(H))^2) across experts; this
script draws such logits (numpy, seeded), adds the bias, counts top-k picks
and bisects alpha until the hottest 35% of experts take the target share.

Run:  python gen/calibrate_zipf.py   (prints alpha; gen.ZIPF_ALPHA_STACK
holds the value used).
"""
import numpy as np


def hot_share(alpha, E=288, k=8, H=6144, tokens=8192, frac=0.35, seed=0):
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((tokens, E)) * (0.05 * np.sqrt(H))
    b = -alpha * np.log(np.arange(1, E + 1))
    top = np.argpartition(-(z + b), k - 1, axis=1)[:, :k]
    counts = np.bincount(top.ravel(), minlength=E)
    n_hot = int(round(frac * E))
    return np.sort(counts)[::-1][:n_hot].sum() / counts.sum()


def calibrate(target=0.74, lo=0.0, hi=4.0, iters=30):
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if hot_share(mid) < target:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


if __name__ == "__main__":
    a = calibrate()
    print(f"alpha = {a:.3f}  hot share = {hot_share(a):.3f}  (66-slot share = "
          f"{hot_share(a, frac=66 / 288):.3f})")
