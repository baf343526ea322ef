"""fp64 numpy oracle for the dense half of the lookup -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU legs may use this module.

Everything is float64; matmul is numpy's (a library primitive). No blocking,
fusion or reordering beyond the formulas:

  projection       v = W_V e_t, k^(m) = W_K^(m) e_t          (Engram notes 3.3/3.4;
                   PageGram report 2.2, W_V in R^{d x 2Kr})
  scalar gate      x <- x + g * v                            (PageGram report 3.1)
  context gate     alpha = sigmoid(RMSNorm(h)^T RMSNorm(k) / sqrt(d))   (Engram notes 3.3,
                   per branch m in 3.4)
  conv + residual  u = alpha v; Y = SiLU(Conv1D_causal(RMSNorm(u))) + u; H <- H + Y
                   (Engram notes 3.3 and 3.1; kernel 4, dilation = max order)

Readings: RMSNorm(z) = z / sqrt(mean(z^2) + eps) * gamma, eps = 1e-6, gamma an
input; the conv is depthwise with weights w[d, 4] shared by the branches and no
bias, c_t = sum_j w[:, j] * z_{t - j*dilation} (tap 0 = current position), with
zeros before the start of the sequence.
"""
from __future__ import annotations

import numpy as np


def project(e: np.ndarray, W: np.ndarray) -> np.ndarray:
    """[n, Din] x [Dout, Din]^T -> [n, Dout]."""
    return np.asarray(e, np.float64) @ np.asarray(W, np.float64).T


def scalar_gate(x: np.ndarray, v: np.ndarray, g: float) -> np.ndarray:
    return np.asarray(x, np.float64) + float(g) * np.asarray(v, np.float64)


def rmsnorm(z: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    z = np.asarray(z, np.float64)
    return z / np.sqrt(np.mean(z * z, axis=-1, keepdims=True) + eps) * np.asarray(gamma, np.float64)


def sigmoid(s: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-np.asarray(s, np.float64)))


def silu(c: np.ndarray) -> np.ndarray:
    c = np.asarray(c, np.float64)
    return c * sigmoid(c)


def context_gate(h: np.ndarray, k: np.ndarray, gamma_h: np.ndarray, gamma_k: np.ndarray,
                 eps: float) -> np.ndarray:
    """alpha over the last axis (d = its length)."""
    d = h.shape[-1]
    s = np.sum(rmsnorm(h, gamma_h, eps) * rmsnorm(k, gamma_k, eps), axis=-1)
    return sigmoid(s / np.sqrt(d))


def engram_gate(e: np.ndarray, W: np.ndarray, h: np.ndarray, gamma_h, gamma_k, eps: float,
                M: int):
    """Multi-branch fusion: W = [W_V; W_K^(1); ...; W_K^(M)] ([(1+M)d, Din]),
    e [n, Din], h [M, n, d] -> (v [n, d], alpha [M, n])."""
    d = W.shape[0] // (1 + M)
    vk = project(e, W)
    v = vk[:, :d]
    alpha = np.stack([context_gate(h[m], vk[:, (1 + m) * d:(2 + m) * d], gamma_h, gamma_k, eps)
                      for m in range(M)])
    return v, alpha


def conv_residual(v: np.ndarray, alpha: np.ndarray, gamma_c: np.ndarray, conv_w: np.ndarray,
                  dilation: int, eps: float, H: np.ndarray) -> np.ndarray:
    """v [B, L, d], alpha [M, B, L], conv_w [d, kernel], H [M, B, L, d] -> H + Y."""
    v = np.asarray(v, np.float64)
    H = np.asarray(H, np.float64)
    w = np.asarray(conv_w, np.float64)
    M = alpha.shape[0]
    B, L, d = v.shape
    out = np.empty_like(H)
    for m in range(M):
        u = np.asarray(alpha[m], np.float64)[..., None] * v
        z = rmsnorm(u, gamma_c, eps)
        c = np.zeros_like(z)
        for j in range(w.shape[1]):
            s = j * dilation
            if s == 0:
                c += w[:, j] * z
            elif s < L:
                c[:, s:, :] += w[:, j] * z[:, :L - s, :]
        out[m] = H[m] + silu(c) + u
    return out
