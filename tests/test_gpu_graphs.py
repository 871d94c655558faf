"""The library's calls inside a CUDA graph.

The library allocates nothing, synchronises nothing, and enqueues everything on the
caller's stream. So forward, backward and decode can be captured once into a CUDA
graph and replayed on new inputs copied into the captured buffers.

Each replay must give what eager calls on the same inputs give:
- bit for bit where the kernels are deterministic: O, LSE, dK, dV and the decode;
- dQ to 1e-5 in relative Frobenius norm, since it is summed by fp32 reductions
  whose order varies.

The eager results themselves are held to the oracle by the other parity tests.
This test also checks one replay against the oracle, on sampled heads.
"""
import pytest
import torch

from oracle import attention_dense_backward
from tests.gpu_util import GRAD_REL_FRO, f64, rel_fro, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_forward_backward_decode_captured_and_replayed():
    from exact_attention_flash_gb300 import (backward_workspace_bytes, decode_workspace_bytes, fa_backward,
                                             fa_decode, fa_device_status, fa_forward)
    from exact_attention_flash_gb300.workloads import make_attention_inputs, make_decode_inputs

    B, H, N, d = 2, 4, 1000, 128
    L, n_split = 5000, 16
    dev = torch.device("cuda")
    x = [t.clone() for t in make_attention_inputs(B, H, N, d, 70, "cuda")]           # q, k, v, do
    xd = [t.clone() for t in make_decode_inputs(B, H, L, d, 71, "cuda")]             # q, k, v
    o = torch.empty_like(x[0])
    lse = torch.empty((B, H, N), device=dev)
    grads32 = [torch.empty(x[0].shape, device=dev) for _ in range(3)]
    grads16 = [torch.empty(x[0].shape, device=dev, dtype=torch.bfloat16) for _ in range(3)]
    ws32 = torch.empty(backward_workspace_bytes(B, H, N, d), device=dev, dtype=torch.uint8)
    ws16 = torch.empty(backward_workspace_bytes(B, H, N, d, torch.bfloat16), device=dev, dtype=torch.uint8)
    od = torch.empty((B, H, 1, d), device=dev)
    lsed = torch.empty((B, H), device=dev)
    wsd = torch.empty(decode_workspace_bytes(B, H, d, n_split), device=dev, dtype=torch.uint8)

    def step():
        q, k, v, do = x
        fa_forward(q, k, v, causal=True, out=o, lse=lse)
        fa_backward(q, k, v, o, lse, do, causal=True, workspace=ws32, dq=grads32[0], dk=grads32[1], dv=grads32[2])
        fa_backward(q, k, v, o, lse, do, causal=True, workspace=ws16, dq=grads16[0], dk=grads16[1], dv=grads16[2],
                    grad_dtype=torch.bfloat16)
        fa_decode(xd[0], xd[1], xd[2], n_split, workspace=wsd, out=od, lse=lsed)

    def results():
        return [t.clone() for t in [o, lse, *grads32, *grads16, od, lsed]]

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    assert fa_device_status() == 0

    for trial in range(3):
        new = make_attention_inputs(B, H, N, d, 80 + trial, "cuda")
        newd = make_decode_inputs(B, H, L, d, 90 + trial, "cuda")
        for dst, src in zip(x + xd, list(new) + list(newd)):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        got = results()
        step()
        torch.cuda.synchronize()
        ref = results()
        assert fa_device_status() == 0
        names = ["O", "LSE", "dQ", "dK", "dV", "dQ bf16", "dK bf16", "dV bf16", "decode O", "decode LSE"]
        for name, g, r in zip(names, got, ref):
            if name.startswith("dQ"):
                assert rel_fro(f64(g), f64(r)) <= 1e-5, name
            else:
                assert torch.equal(g, r), name
        if trial == 0:
            q, k, v, do = x
            for b, h in [(0, 1), (1, 3)]:
                r = attention_dense_backward(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), f64(do[b, h]), causal=True)
                for gname, gg, rr in zip(("dQ", "dK", "dV"), (t[b, h] for t in got[2:5]), r):
                    assert rel_fro(f64(gg), rr) <= GRAD_REL_FRO, gname



def test_two_captured_forwards_replayed_concurrently_on_two_streams():
    """Two forwards captured into two graphs, each with its own workspace (the
    persistent grid's work counter) and outputs, replayed at the same time on two
    streams. The small problem's grid takes a few SMs while the large one's fills
    the rest, so the two grids run side by side and claim work items at the same
    time. Each result must equal an eager call on the same inputs bit for bit: no
    item is lost or computed twice."""
    from exact_attention_flash_gb300 import fa_forward, fa_get_device_status, forward_workspace_bytes
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    shapes = [(2, 16, 4096, 128, True), (1, 4, 2048, 64, False)]
    runs = []
    for i, (B, H, N, d, causal) in enumerate(shapes):
        q, k, v, _ = make_attention_inputs(B, H, N, d, 400 + i, "cuda", with_do=False)
        ref_o, ref_l = fa_forward(q, k, v, causal=causal)
        o = torch.empty_like(ref_o)
        lse = torch.empty_like(ref_l)
        ws = torch.empty(forward_workspace_bytes(B, H, N, d, causal), device="cuda", dtype=torch.uint8)
        runs.append(dict(q=q, k=k, v=v, causal=causal, o=o, lse=lse, ws=ws, ref=(ref_o, ref_l)))
    torch.cuda.synchronize()

    streams = [torch.cuda.Stream() for _ in runs]
    graphs = []
    for r, s in zip(runs, streams):
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):  # warm-up outside the capture
            fa_forward(r["q"], r["k"], r["v"], causal=r["causal"], out=r["o"], lse=r["lse"], workspace=r["ws"])
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fa_forward(r["q"], r["k"], r["v"], causal=r["causal"], out=r["o"], lse=r["lse"], workspace=r["ws"])
        graphs.append(g)
    torch.cuda.synchronize()

    for trial in range(20):
        for r in runs:
            r["o"].fill_(float("nan"))
            r["lse"].fill_(float("nan"))
        torch.cuda.synchronize()
        order = [1, 0] if trial % 2 == 0 else [0, 1]
        for i in order:
            with torch.cuda.stream(streams[i]):
                graphs[i].replay()
        torch.cuda.synchronize()
        assert fa_get_device_status() == 0
        for i, r in enumerate(runs):
            assert torch.equal(r["o"], r["ref"][0]), (trial, i, "O")
            assert torch.equal(r["lse"], r["ref"][1]), (trial, i, "LSE")
