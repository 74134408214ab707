"""Unsharded MLP block in float64: the plain definition the sharded GPU path
must reproduce.

Source: page "一层 MLP 太宽而放不下时怎样切？" (zwjcode.cn), §01 (H = act(X W1),
Y = H W2), §05 (b2 added once; b1 follows the columns), §06 (backward:
dW2 and dH local, dX = sum over column shards of dZ W1^T). The activation is
ReLU, the tanh form of GELU (Hendrycks & Gimpel, "Gaussian Error Linear
Units", 2016: 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))), or the exact
(erf) GELU the pages' code uses (`nn.GELU()`, `F.gelu`, §01 and the course
notes' FFN): z Phi(z) = 0.5 z (1 + erf(z / sqrt(2))), Phi the standard normal
CDF; its derivative is Phi(z) + z phi(z), phi the standard normal density;
or the sigmoid approximation of GELU on the interview page (`x / (1 +
exp(-1.702 x))`): z s(z), s = sigmoid(1.702 z), derivative s (1 + 1.702 z (1 - s)).

Conventions taken where the pages are silent:
- ReLU'(0) = 0 (strict z > 0), the usual autograd convention;
- GELU' is the exact derivative of the tanh form above.
"""

import math

import numpy as np
from scipy.special import erf

SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
GELU_CUBIC = 0.044715
GELU_SIGMOID_SCALE = 1.702


def as_f64(a):
    """Promote a torch tensor or array-like to a float64 numpy array (exact
    for fp32 and bf16 inputs)."""
    if a is None:
        return None
    if hasattr(a, "detach"):
        return a.detach().to("cpu").double().numpy()
    return np.asarray(a, dtype=np.float64)


def act(z, kind):
    z = np.asarray(z, dtype=np.float64)
    if kind == "relu":
        return np.where(z > 0.0, z, 0.0)
    if kind == "gelu_tanh":
        u = SQRT_2_OVER_PI * (z + GELU_CUBIC * z ** 3)
        return 0.5 * z * (1.0 + np.tanh(u))
    if kind == "gelu_erf":
        return 0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))
    if kind == "gelu_sigmoid":
        return z / (1.0 + np.exp(-GELU_SIGMOID_SCALE * z))
    raise ValueError(kind)


def act_grad(z, kind):
    """d act / dz evaluated at z."""
    z = np.asarray(z, dtype=np.float64)
    if kind == "relu":
        return np.where(z > 0.0, 1.0, 0.0)
    if kind == "gelu_tanh":
        u = SQRT_2_OVER_PI * (z + GELU_CUBIC * z ** 3)
        t = np.tanh(u)
        du = SQRT_2_OVER_PI * (1.0 + 3.0 * GELU_CUBIC * z ** 2)
        return 0.5 * (1.0 + t) + 0.5 * z * (1.0 - t * t) * du
    if kind == "gelu_erf":
        cdf = 0.5 * (1.0 + erf(z / math.sqrt(2.0)))
        pdf = np.exp(-0.5 * z * z) / math.sqrt(2.0 * math.pi)
        return cdf + z * pdf
    if kind == "gelu_sigmoid":
        sg = 1.0 / (1.0 + np.exp(-GELU_SIGMOID_SCALE * z))
        return sg * (1.0 + GELU_SIGMOID_SCALE * z * (1.0 - sg))
    raise ValueError(kind)


def forward(X, W1, b1, W2, b2, kind):
    """Y = act(X W1 + b1) W2 + b2 with the full W1 [D, F], W2 [F, D].

    Returns dict(Z=[N, F], H=[N, F], Y=[N, D]). Each output row depends only
    on the same row of X, so forward(X[rows], ...) gives exactly those rows."""
    X, W1, W2 = as_f64(X), as_f64(W1), as_f64(W2)
    Z = X @ W1
    if b1 is not None:
        Z = Z + as_f64(b1)[None, :]
    H = act(Z, kind)
    Y = H @ W2
    if b2 is not None:
        Y = Y + as_f64(b2)[None, :]
    return {"Z": Z, "H": H, "Y": Y}


def backward(X, W1, b1, W2, dY, kind):
    """Gradients of <dY, Y> for Y = act(X W1 + b1) W2 + b2.

    Returns dict(dH, dZ, dX=[N, D], dW1=[D, F], dW2=[F, D], db1=[F], db2=[D]).
    The forward quantities are recomputed here from the inputs, so the
    result never depends on a saved (and possibly rounded) Z or H.

    Separability used by the sampled checks: hidden unit f only touches
    W1[:, f], b1[f], W2[f, :], so backward on the columns fidx of W1 (and
    rows fidx of W2) returns exactly dW1[:, fidx], dW2[fidx, :], db1[fidx];
    and dX row n depends only on rows n of X and dY."""
    X, W1, W2, dY = as_f64(X), as_f64(W1), as_f64(W2), as_f64(dY)
    Z = X @ W1
    if b1 is not None:
        Z = Z + as_f64(b1)[None, :]
    H = act(Z, kind)
    dH = dY @ W2.T
    dZ = dH * act_grad(Z, kind)
    return {
        "dH": dH,
        "dZ": dZ,
        "dX": dZ @ W1.T,
        "dW1": X.T @ dZ,
        "dW2": H.T @ dY,
        "db1": dZ.sum(axis=0),
        "db2": dY.sum(axis=0),
    }


def forward_rows(X, W1, b1, W2, b2, kind, rows):
    """Rows `rows` of forward(): the definition applied to those tokens."""
    X = as_f64(X)
    return forward(X[np.asarray(rows)], W1, b1, W2, b2, kind)


def backward_rows_dx(X, W1, b1, W2, dY, kind, rows):
    """Rows `rows` of dX (each dX row needs only that token's X and dY)."""
    rows = np.asarray(rows)
    return backward(as_f64(X)[rows], W1, b1, W2, as_f64(dY)[rows], kind)["dX"]


def backward_hidden_units(X, W1, b1, W2, dY, kind, fidx):
    """dW1[:, fidx], dW2[fidx, :] and db1[fidx] over ALL tokens, computed on
    the sub-block that keeps only hidden units `fidx`."""
    fidx = np.asarray(fidx)
    W1s = as_f64(W1)[:, fidx]
    W2s = as_f64(W2)[fidx, :]
    b1s = None if b1 is None else as_f64(b1)[fidx]
    g = backward(X, W1s, b1s, W2s, dY, kind)
    return {"dW1": g["dW1"], "dW2": g["dW2"], "db1": g["db1"]}


def silu(z):
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def swiglu_forward(X, Wg, Wu, Wd):
    """Gated MLP of page "一层 MLP 太宽而放不下时怎样切？" §08:
    G = X Wg, U = X Wu, H = SiLU(G) * U, Y = H Wd, with Wg, Wu [D, F] and
    Wd [F, D] unsharded. SiLU(z) = z / (1 + exp(-z))."""
    X, Wg, Wu, Wd = as_f64(X), as_f64(Wg), as_f64(Wu), as_f64(Wd)
    G = X @ Wg
    U = X @ Wu
    H = silu(G) * U
    return {"G": G, "U": U, "H": H, "Y": H @ Wd}
