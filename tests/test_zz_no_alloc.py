"""tpmlp_forward_noalloc against the existing tpmlp_forward, through the C-ABI.

Some callers of this library cannot allocate device memory on the forward
path: a plug-in running inside a host program that owns every byte of device
memory, or a latency-bound loop that may not risk a cudaMalloc (it can fail
or synchronise the device). tpmlp_forward_noalloc serves them: it runs the
PARTIALS forward with the T fp32 partial sums in a fixed 8 MiB array inside
the library, so the caller passes only inputs and outputs.

The test makes two calls in a row (different shapes, dtypes and inputs, so
the second call finds the first call's partials still in the shared array)
and compares each with tpmlp_forward in PARTIALS mode, within the parity
tolerance of the dtype. It runs alone or after the other tests.
"""

import pytest
import torch

import tensor_transformer_mlp_columnparallel_gb300 as tp
from tensor_transformer_mlp_columnparallel_gb300 import _binding
from tests.gpu_helpers import to_gpu
from tests.tolerance import normwise_rel_err, TOL
from workloads.gen import gen_random_mlp

pytestmark = pytest.mark.gpu

SCRATCH = 8 << 20   # TPMLP_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _outputs(inp, dev):
    dt = inp.X.dtype
    Y = torch.empty(inp.N, inp.D, dtype=dt, device=dev)
    H = [torch.empty(inp.N, inp.Fs, dtype=dt, device=dev) for _ in range(inp.T)]
    Z = [torch.empty(inp.N, inp.Fs, dtype=dt, device=dev) for _ in range(inp.T)]
    return Y, H, Z


def test_noalloc_forward_matches_forward_on_two_calls_in_a_row():
    dev = torch.device("cuda:0")
    cases = [
        # T * N * D * 4 = 8 MiB: the largest shape the array takes
        dict(N=64, D=4096, F=4096, T=8, dtype="bf16", act="gelu_tanh", bias=True, seed=101),
        # a smaller fp32 call that lands on the first call's leftovers
        dict(N=40, D=264, F=4 * 136, T=4, dtype="f32", act="relu", bias=True, seed=102),
    ]
    for c in cases:
        inp = gen_random_mlp(with_dy=False, **c)
        assert inp.T * ((inp.N * inp.D * 4 + 255) // 256 * 256) <= SCRATCH
        g = to_gpu(inp)
        Yr, Hr, Zr = tp.mlp_forward(g["X"], g["W1"], g["W2"], g["b1"], g["b2"], act=c["act"],
                                    mode="partials")
        Y, H, Z = _outputs(inp, dev)
        tp.tpmlp_forward_noalloc(g["X"], g["W1"], g["b1"], g["W2"], g["b2"], Y, H, Z, c["act"])
        torch.cuda.synchronize()
        tol = TOL[c["dtype"]]
        assert normwise_rel_err(Y, Yr) <= tol
        for r in range(inp.T):
            assert normwise_rel_err(H[r], Hr[r]) <= tol
            assert normwise_rel_err(Z[r], Zr[r]) <= tol
    assert tp.tpmlp_check_device_error() == 0


def test_noalloc_forward_rejects_shapes_beyond_its_array():
    dev = torch.device("cuda:0")
    inp = gen_random_mlp(N=65, D=4096, F=4096, T=8, dtype="bf16", act="gelu_tanh", bias=False,
                         seed=103, with_dy=False)
    g = to_gpu(inp)
    Y, H, Z = _outputs(inp, dev)
    before = tp.tpmlp_launch_count()
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_forward_noalloc(g["X"], g["W1"], None, g["W2"], None, Y, H, Z, "gelu_tanh")
    assert e.value.status == _binding.ERR_WORKSPACE
    assert tp.tpmlp_launch_count() == before
