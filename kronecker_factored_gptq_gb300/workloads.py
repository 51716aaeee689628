"""Seeded synthetic inputs for the BaKron solver.

This module only draws random numbers and forms Gram matrices; it holds none
of the solver's arithmetic (no damping, no factorisation, no quantisation) and
is the one module that both the CUDA path's callers and the CPU oracle's
callers use to get identical inputs.

Each workload returns fp32 arrays: the weight ``W`` (m x n), the raw input-side
factor ``A`` (n x n) and output-side factor ``B`` (m x m) BEFORE damping, the
damping fractions the solver's preparation step adds, and the grid.  The
recipes follow the five workloads the solver is specified on; the pages
measure runtime on plain matrix shapes with no dataset (summary page "FastKron:
Efficient Quantization with Kronecker-Factored Hessians", Table 3: 8192 x 8192;
ainews article on BaKron: 4096 x 14336 and its transpose), so these synthetic
matrices stand in for real layer weights and activation statistics.

Random streams: ``np.random.default_rng([seed, k])`` with a fixed k per
component, so components do not shift when another one changes.  Gram
matrices ``X X^T / N`` are formed in fp64 (numpy on the host, or torch on a
given device for the large ones) and rounded once to fp32.
"""

from dataclasses import dataclass, field

import numpy as np


@dataclass
class Workload:
    name: str
    m: int
    n: int
    W: np.ndarray          # m x n fp32
    A: np.ndarray          # n x n fp32, input side, undamped
    B: np.ndarray          # m x m fp32, output side, undamped
    damp_A: float
    damp_B: float
    bits: int
    qmin: int
    qmax: int
    desc: str = ""
    extra: dict = field(default_factory=dict)


def _rng(seed, k):
    return np.random.default_rng([int(seed), int(k)])


def _gram(X, N, device=None):
    """``X X^T / N`` in fp64, returned as fp32."""
    if device is not None and str(device) != "cpu":
        import torch
        Xt = torch.from_numpy(np.ascontiguousarray(X, dtype=np.float64)).to(device)
        G = (Xt @ Xt.T) / float(N)
        return G.to(torch.float32).cpu().numpy()
    X = np.asarray(X, dtype=np.float64)
    return ((X @ X.T) / float(N)).astype(np.float32)


def _haar_orthogonal(rng, k):
    """Haar-distributed orthogonal k x k matrix (QR of a Gaussian, sign-fixed)."""
    Z = rng.standard_normal((k, k))
    Q, R = np.linalg.qr(Z)
    return Q * np.sign(np.diag(R))[None, :]


def _ar1_rows(rng, rows, cols, rho):
    """Rows of an AR(1) process along the row index: x_0 = z_0,
    x_t = rho x_{t-1} + sqrt(1 - rho^2) z_t (stationary covariance rho^|t-t'|)."""
    X = rng.standard_normal((rows, cols))
    c = np.sqrt(1.0 - rho * rho)
    for t in range(1, rows):
        X[t] = rho * X[t - 1] + c * X[t]
    return X


def _grid(bits):
    qmax = (1 << (bits - 1)) - 1
    return bits, -(qmax + 1), qmax


def tiny64(seed=0, device=None):
    """64 x 64; W ~ N(0, 0.02^2); A = X X^T/512, B = G G^T/512 with X, G 64 x 512
    standard normal; 1% damping on both; 4-bit grid [-8, 7]."""
    m = n = 64
    W = (0.02 * _rng(seed, 1).standard_normal((m, n))).astype(np.float32)
    A = _gram(_rng(seed, 2).standard_normal((n, 512)), 512, device)
    B = _gram(_rng(seed, 3).standard_normal((m, 512)), 512, device)
    return Workload("tiny64", m, n, W, A, B, 0.01, 0.01, *_grid(4),
                    desc="64x64, 4-bit, Gaussian Gram factors")


def c1024(seed=0, device=None):
    """1024 x 1024; A from X (1024 x 4096) with log-normal(0, 1) channel
    scales; B from O G with G (1024 x 4096) standard normal and O Haar
    orthogonal; 1% damping on both; 4-bit grid."""
    m = n = 1024
    W = (0.02 * _rng(seed, 1).standard_normal((m, n))).astype(np.float32)
    r = _rng(seed, 2)
    scales = np.exp(r.standard_normal(n))
    X = scales[:, None] * r.standard_normal((n, 4096))
    A = _gram(X, 4096, device)
    r = _rng(seed, 3)
    G = r.standard_normal((m, 4096))
    O = _haar_orthogonal(_rng(seed, 4), m)
    B = _gram(O @ G, 4096, device)
    return Workload("c1024", m, n, W, A, B, 0.01, 0.01, *_grid(4),
                    desc="1024x1024, 4-bit, log-normal channel scales, rotated B")


def c4096(seed=0, device=None):
    """4096 x 4096; W ~ Student-t(5) * 0.02; A = AR(1) covariance rho = 0.9
    (A_jk = 0.9^|j-k|); B = G G^T/8192 with G (4096 x 8192); 1% damping on
    both; 3-bit grid [-4, 3]."""
    m = n = 4096
    W = (0.02 * _rng(seed, 1).standard_t(5, size=(m, n))).astype(np.float32)
    idx = np.arange(n)
    A = (0.9 ** np.abs(idx[:, None] - idx[None, :])).astype(np.float32)
    B = _gram(_rng(seed, 3).standard_normal((m, 8192)), 8192, device)
    return Workload("c4096", m, n, W, A, B, 0.01, 0.01, *_grid(3),
                    desc="4096x4096, 3-bit, Student-t weights, AR(1) A")


def mlp(m, n, seed=0, device=None):
    """MLP projection shape; W ~ N(0, 0.015^2); A = X X^T/16384 with X
    (n x 16384) standard normal and floor(n/100) channels scaled x20, NO
    damping on A; B = G G^T/16384 with G (m x 16384), 1% damping; 4-bit."""
    W = (0.015 * _rng(seed, 1).standard_normal((m, n))).astype(np.float32)
    r = _rng(seed, 2)
    X = r.standard_normal((n, 16384))
    out = r.choice(n, size=n // 100, replace=False)
    X[out] *= 20.0
    A = _gram(X, 16384, device)
    del X
    B = _gram(_rng(seed, 3).standard_normal((m, 16384)), 16384, device)
    return Workload("mlp%dx%d" % (m, n), m, n, W, A, B, 0.0, 0.01, *_grid(4),
                    desc="%dx%d MLP projection, 4-bit, 1%% outlier channels x20, undamped A" % (m, n))


def c8192(seed=0, device=None):
    """8192 x 8192 (the headline shape); A = X X^T/16384 with X (8192 x 16384)
    AR(1) rho = 0.95 across channels, 1% damping; B = G G^T/2048 with G
    (8192 x 2048), rank 2048, made definite by 1% damping; 2-bit [-2, 1]."""
    m = n = 8192
    W = (0.02 * _rng(seed, 1).standard_normal((m, n))).astype(np.float32)
    X = _ar1_rows(_rng(seed, 2), n, 16384, 0.95)
    A = _gram(X, 16384, device)
    del X
    B = _gram(_rng(seed, 3).standard_normal((m, 2048)), 2048, device)
    return Workload("c8192", m, n, W, A, B, 0.01, 0.01, *_grid(2),
                    desc="8192x8192, 2-bit, AR(1) A, rank-deficient B")


def random_problem(m, n, seed=0, bits=4, damp=0.01, oversample=2, device=None):
    """Generic m x n case for parity tests at arbitrary (ragged) sizes:
    W ~ N(0, 0.02^2), A = X X^T/N, B = G G^T/N with N = oversample * size."""
    W = (0.02 * _rng(seed, 11).standard_normal((m, n))).astype(np.float32)
    Na = max(1, oversample * n)
    Nb = max(1, oversample * m)
    A = _gram(_rng(seed, 12).standard_normal((n, Na)), Na, device)
    B = _gram(_rng(seed, 13).standard_normal((m, Nb)), Nb, device)
    return Workload("rand%dx%d" % (m, n), m, n, W, A, B, damp, damp, *_grid(bits),
                    desc="random %dx%d" % (m, n))


CONFIGS = {
    "tiny64": tiny64,
    "c1024": c1024,
    "c4096": c4096,
    "mlp4096x14336": lambda seed=0, device=None: mlp(4096, 14336, seed, device),
    "mlp14336x4096": lambda seed=0, device=None: mlp(14336, 4096, seed, device),
    "c8192": c8192,
}


def load(name, seed=0, device=None):
    return CONFIGS[name](seed=seed, device=device)


def sample_stream(N, n, m, seed=0):
    """N samples of a layer's input activations (N x n, channel scales drawn
    log-normal(0, 1) as in the 1024 x 1024 workload) and output gradients
    (N x m, standard normal), fp32: the inputs of the Kronecker-factor
    accumulation."""
    rng = _rng(seed, 20)
    X = rng.standard_normal((N, n), dtype=np.float32)
    X *= np.exp(_rng(seed, 21).standard_normal(n)).astype(np.float32)[None, :]
    G = _rng(seed, 22).standard_normal((N, m), dtype=np.float32)
    return X, G
