"""Error bounds for the kernels' fp32 activations (test infrastructure).

The kernels evaluate GeLU, SiLU and QGeLU (and their derivatives) in fp32 as
x * sigmoid(t), with sigmoid(t) formed from e = 2^(-|t| log2 e) by the hardware
ex2 / rcp approximations; the oracle evaluates the same expressions exactly in
double.  Two sources of error in the fp32 evaluation:

  - the approximations and the fp32 roundings of the arithmetic: a few fp32
    ulps of the result, bounded here by DELTA = 2^-20 (8 ulps);
  - the rounding of the argument t itself (its fp32 evaluation carries a
    relative error of a few 2^-24), which exp magnifies by |t|: the relative
    error of sigmoid(t) with respect to a relative error in t is
    |t| * sigmoid(-t).  Any fp32 evaluation has this term, whatever its exp.

So the kernels' act(x) must satisfy |gpu - exact| <= DELTA * cond * |exact|
with cond = 1 + |t| sigmoid(-t); and act'(x) = s (1 + q) (s = sigmoid(t),
q = x (1 - s) t') must satisfy |gpu - exact| <= DELTA (1 + |t|) |s| (|1 + q| + |q|):
relative to the size of the terms the evaluation adds, so where act' crosses
zero (1 + q -> 0) the bound relative to the result grows with the condition
number 1 + |q| / |1 + q|.  Results in fp32's subnormal range get SUB more.
"""
import numpy as np

DELTA = 2.0 ** -20
SUB = 2.0 ** -147
C_GELU = 1.5957691216057308      # 2 sqrt(2 / pi)


def sigmoid_arg(xv, act):
    return {3: C_GELU * (xv + 0.044715 * xv ** 3), 4: xv, 5: 1.702 * xv}[act]


def _sig(t):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-t))


def forward_cond(xv, act):
    """cond for act(x): 1 + |t| sigmoid(-t)."""
    t = sigmoid_arg(xv, act)
    return 1.0 + np.abs(t) * _sig(-t)


def derivative_terms(xv, act):
    """(1 + |t|) |s| (|1 + q| + |q|) for act'(x) = s (1 + q)."""
    t = sigmoid_arg(xv, act)
    s, oms = _sig(t), _sig(-t)
    tp = {3: C_GELU * (1.0 + 3 * 0.044715 * xv ** 2), 4: np.ones_like(xv), 5: np.full_like(xv, 1.702)}[act]
    q = xv * oms * tp
    return (1.0 + np.abs(t)) * np.abs(s) * (np.abs(1.0 + q) + np.abs(q))


def derivative_cond(xv, act, exact):
    """cond for act'(x) relative to |act'(x)| (exact: the oracle's act'(x) in double)."""
    with np.errstate(divide="ignore", invalid="ignore"):
        return derivative_terms(xv, act) / np.maximum(np.abs(exact), 1e-300)
