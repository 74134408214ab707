"""Error metrics and tolerances shared by the parity tests.

Normwise max relative error of a result g against the oracle o (one output
tensor at a time):  max_i |g_i - o_i| / max_i |o_i|.

Tolerances: 1e-5 when the path stores and computes in fp32, 2e-2 when it
stores bf16 and accumulates in fp32.
"""

import numpy as np

TOL = {"f32": 1e-5, "bf16": 2e-2}


def to_f64(a):
    if hasattr(a, "detach"):
        return a.detach().to("cpu").double().numpy()
    return np.asarray(a, dtype=np.float64)


def normwise_rel_err(got, ref):
    g, o = to_f64(got), to_f64(ref)
    assert g.shape == o.shape, (g.shape, o.shape)
    if o.size == 0:
        return 0.0
    denom = np.max(np.abs(o))
    diff = np.max(np.abs(g - o))
    if denom == 0.0:
        return float(diff)
    return float(diff / denom)


def assert_close(got, ref, dtype, what=""):
    err = normwise_rel_err(got, ref)
    tol = TOL[dtype]
    assert err <= tol, f"{what}: normwise rel err {err:.3e} > {tol:.1e}"
    return err
