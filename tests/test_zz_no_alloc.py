"""tpmlp_forward_noalloc through the C-ABI: against the float64 oracle, and
against the existing tpmlp_forward given a workspace of the same size.

Some callers of this library cannot allocate device memory on the forward
path: a plug-in running inside a host program that owns every byte of device
memory, or a latency-bound loop that may not risk a cudaMalloc (it can fail
or synchronise the device). tpmlp_forward_noalloc serves them: it runs the
PARTIALS forward with the T fp32 partial sums (and, where they fit behind
them, the few-token GEMMs' stream-K counters and partial slots) in a fixed
8 MiB array inside the library, so the caller passes only inputs and outputs.

The cases run two calls in a row each, so every call finds the previous
call's partial sums and counters still in the shared array; each result is
compared with the oracle within the parity tolerance of its dtype, and bit
for bit with tpmlp_forward in PARTIALS mode given a caller workspace of
exactly TPMLP_NOALLOC_SCRATCH_BYTES (the same sizes give the same launch
plans). A warm call must leave the device's free memory unchanged. The file
runs alone or after the other tests.
"""

import pytest
import torch

import oracle
import tensor_transformer_mlp_columnparallel_gb300 as tp
from tensor_transformer_mlp_columnparallel_gb300 import _binding
from tests.gpu_helpers import to_gpu
from tests.tolerance import assert_close
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


def _check_case(c, dev):
    """Two noalloc calls of one case, each against the oracle and bit for bit
    against tpmlp_forward with an 8 MiB caller workspace."""
    inp = gen_random_mlp(with_dy=False, **c)
    assert inp.T * ((inp.N * inp.D * 4 + 255) // 256 * 256) <= SCRATCH
    g = to_gpu(inp)
    ws = torch.empty(SCRATCH, dtype=torch.uint8, device=dev)
    Yr, Hr, Zr = _outputs(inp, dev)
    tp.tpmlp_forward(g["X"], g["W1"], g["b1"], g["W2"], g["b2"], Yr, Hr, Zr, c["act"], "partials",
                     ws)
    f = oracle.mlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, c["act"])
    for _ in range(2):
        Y, H, Z = _outputs(inp, dev)
        tp.tpmlp_forward_noalloc(g["X"], g["W1"], g["b1"], g["W2"], g["b2"], Y, H, Z, c["act"])
        torch.cuda.synchronize()
        assert_close(Y, f["Y"], c["dtype"], "Y")
        assert_close(torch.cat([h.float() for h in H], 1), f["H"], c["dtype"], "H")
        assert_close(torch.cat([z.float() for z in Z], 1), f["Z"], c["dtype"], "Z")
        assert torch.equal(Y, Yr)
        for r in range(inp.T):
            assert torch.equal(H[r], Hr[r]) and torch.equal(Z[r], Zr[r])


def test_noalloc_forward_matches_oracle_and_forward_on_two_calls_in_a_row():
    dev = torch.device("cuda:0")
    # T * N * D * 4 = 8 MiB: the largest shape the array takes (no room for
    # the stream-K scratch behind the partials)
    _check_case(dict(N=64, D=4096, F=4096, T=8, dtype="bf16", act="gelu_tanh", bias=True,
                     seed=101), dev)
    # a smaller fp32 call that lands on the first call's leftovers
    _check_case(dict(N=40, D=264, F=4 * 136, T=4, dtype="f32", act="relu", bias=True, seed=102),
                dev)
    assert tp.tpmlp_check_device_error() == 0


def test_noalloc_forward_few_tokens_runs_stream_k_inside_the_array():
    """8 tokens, D = 2048, F = 256, T = 2: the partials take 128 KB of the
    array and the stream-K counters and partial slots (about 4 MiB) fit
    behind them, so the column GEMM (two tiles, 32 k-blocks each) runs in the
    stream-K form out of the library's array. Its counters are reset on the
    stream before each launch; the second call finds the first call's counts
    there."""
    dev = torch.device("cuda:0")
    assert tp.tpmlp_gemm_plan(8, 128, 2048, 2, balanced=True)[2] == 0
    need = tp.tpmlp_workspace_bytes_balanced(_binding.OP_FORWARD, torch.bfloat16, 8, 2048, 256,
                                             2, "partials")
    assert need <= SCRATCH
    _check_case(dict(N=8, D=2048, F=256, T=2, dtype="bf16", act="gelu_tanh", bias=True, seed=104),
                dev)
    assert tp.tpmlp_check_device_error() == 0


def test_noalloc_forward_allocates_no_device_memory():
    dev = torch.device("cuda:0")
    inp = gen_random_mlp(N=16, D=1024, F=2048, T=4, dtype="bf16", act="gelu_tanh", bias=True,
                         seed=105, with_dy=False)
    g = to_gpu(inp)
    Y, H, Z = _outputs(inp, dev)
    call = lambda: tp.tpmlp_forward_noalloc(g["X"], g["W1"], g["b1"], g["W2"], g["b2"], Y, H, Z,
                                            "gelu_tanh")
    call()   # a warm call: the library's module and its static array are resident
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info(dev)[0]
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(dev)[0] == free0
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
