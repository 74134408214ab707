"""The library's launches captured into a CUDA graph and replayed.

Every entry point launches on the caller's stream and keeps no host state
between calls that a replay would miss (tensor maps and kernel parameters are
passed by value at launch), so a forward + backward step, or a CE forward and
backward, captured once and replayed, must give bit-identical results to the
same calls made eagerly: all kernels are deterministic. The shapes cover the
CTA-pair GEMM, the K-split GEMM (a few token rows), the stream-K GEMM (a few
token rows with the scratch: a counter reset and a launch per GEMM, partial
tiles summed in CTA order), the fp32 CUDA-core GEMM and both block-end modes.
"""

import pytest
import torch

import tensor_transformer_mlp_columnparallel_gb300 as tp
from tensor_transformer_mlp_columnparallel_gb300 import _binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert tp.tpmlp_check_device_error() == 0


def dev():
    return torch.device("cuda:0")


def block_buffers(N, D, F, T, dtype, mode, seed, balanced=False):
    g = torch.Generator(device=dev())
    g.manual_seed(seed)
    Fs = F // T
    r = lambda *s, sc=1.0: (torch.randn(*s, generator=g, device=dev()) * sc).to(dtype)
    b = {
        "X": r(N, D), "dY": r(N, D),
        "W1": [r(D, Fs, sc=D ** -0.5) for _ in range(T)],
        "W2": [r(Fs, D, sc=F ** -0.5) for _ in range(T)],
        "Y": torch.empty(N, D, dtype=dtype, device=dev()),
        "H": [torch.empty(N, Fs, dtype=dtype, device=dev()) for _ in range(T)],
        "Z": [torch.empty(N, Fs, dtype=dtype, device=dev()) for _ in range(T)],
        "dX": torch.empty(N, D, dtype=dtype, device=dev()),
        "dW1": [torch.empty(D, Fs, dtype=dtype, device=dev()) for _ in range(T)],
        "dW2": [torch.empty(Fs, D, dtype=dtype, device=dev()) for _ in range(T)],
    }
    size = tp.tpmlp_workspace_bytes_balanced if balanced else tp.tpmlp_workspace_bytes
    wf = size(_binding.OP_FORWARD, dtype, N, D, F, T, mode)
    wb = size(_binding.OP_BACKWARD, dtype, N, D, F, T, mode)
    b["ws"] = torch.empty(max(wf, wb, 256), dtype=torch.uint8, device=dev())
    return b


def step(b, mode):
    tp.tpmlp_forward(b["X"], b["W1"], None, b["W2"], None, b["Y"], b["H"], b["Z"], "gelu_tanh",
                     mode, b["ws"])
    tp.tpmlp_backward(b["X"], b["W1"], b["W2"], b["H"], b["Z"], b["dY"], b["dX"], b["dW1"],
                      b["dW2"], None, None, "gelu_tanh", mode, b["ws"])


def outputs(b):
    return [t.clone() for t in [b["Y"], b["dX"], *b["H"], *b["dW1"], *b["dW2"]]]


@pytest.mark.parametrize("N,D,F,T,dtype,mode,balanced", [
    (512, 512, 2048, 2, torch.bfloat16, "splitk", False),      # CTA-pair tiles
    (16, 1024, 8192, 4, torch.bfloat16, "splitk", False),      # K-split row and dX GEMMs
    (16, 1024, 8192, 4, torch.bfloat16, "partials", False),    # partial sums + block-end reduce
    (16, 1024, 8192, 4, torch.bfloat16, "splitk", True),       # stream-K GEMMs
    (40, 2048, 8000, 4, torch.bfloat16, "partials", True),     # stream-K, 64-row slots
    (64, 256, 1024, 2, torch.float32, "splitk", False),        # fp32 CUDA-core GEMM
])
def test_graph_replay_matches_eager_bit_for_bit(N, D, F, T, dtype, mode, balanced):
    b = block_buffers(N, D, F, T, dtype, mode, seed=N + D + T, balanced=balanced)
    step(b, mode)                     # eager (also loads modules, sets kernel attributes)
    torch.cuda.synchronize()
    want = outputs(b)
    for t in [b["Y"], b["dX"], *b["H"], *b["dW1"], *b["dW2"]]:
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(b, mode)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    got = outputs(b)
    for w, g_ in zip(want, got):
        assert torch.equal(w, g_)


def test_graph_replay_of_cross_entropy_forward_and_backward():
    N, V, T = 256, 16000, 8
    g = torch.Generator(device=dev())
    g.manual_seed(3)
    logits = torch.randn(N, V, generator=g, device=dev()) * 2
    targets = torch.randint(0, V, (N,), generator=g, device=dev())
    loss = torch.empty(N, device=dev())
    mean = torch.empty(1, device=dev())
    amax = torch.empty(N, dtype=torch.int32, device=dev())
    own = torch.empty(N, dtype=torch.int32, device=dev())
    dlog = torch.empty_like(logits)

    def run():
        tp.tpmlp_vocab_ce(logits, targets, T, loss, mean, amax, own)
        tp.tpmlp_vocab_ce_backward(logits, targets, T, loss, 1.0 / N, dlog)

    run()
    torch.cuda.synchronize()
    want = [loss.clone(), mean.clone(), amax.clone(), own.clone(), dlog.clone()]
    for t in (loss, mean, dlog):
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    graph.replay()
    torch.cuda.synchronize()
    for w, g_ in zip(want, [loss, mean, amax, own, dlog]):
        assert torch.equal(w, g_)
