"""Re-derivation of the 16 NormalFloat-4 levels held as a literal table by the C oracle.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The PageGram report stores deployed rows as NF4 (QLoRA's data type, section 3.3) but
prints no level values; the oracle holds the values the QLoRA paper prints (Dettmers et
al. 2023, Appendix E). This module restates the construction behind them as a check:
levels are quantiles of the standard normal at evenly spaced probabilities, with an exact
zero, 7 strictly negative and 8 strictly positive levels (an asymmetric type), the
outermost probability on each side being delta = 1 - (1/30 + 1/32)/2 (a quantile at
probability 1 would be infinite), scaled so the extremes are -1, +1. Computed in fp64
with this exact delta it lands within 2 fp32 ulps (<= 1.8e-7) of the printed values,
which were computed with delta rounded to 0.9677083 and fp32 probability grids.
"""
import numpy as np


def derive_levels() -> np.ndarray:
    from scipy.stats import norm

    delta = 1.0 - 0.5 * (1.0 / 30.0 + 1.0 / 32.0)
    pos = norm.ppf(np.linspace(delta, 0.5, 9)[:-1])       # 8 positive levels
    neg = -norm.ppf(np.linspace(delta, 0.5, 8)[:-1])      # 7 negative levels
    v = np.sort(np.concatenate([neg, [0.0], pos]))
    return (v / v.max()).astype(np.float32)


if __name__ == "__main__":
    for x in derive_levels():
        print(f"0x{np.float32(x).view(np.uint32):08x}u  /* {float(x)!r} */")
