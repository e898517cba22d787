"""The C ABI under CUDA graph capture, as a serving loop runs it: decode steps,
kda_decode_tokens and the prefill plans (including the windowed plan's side
stream, which joins the capture through events) captured once and replayed on
new inputs copied into the same buffers; every replay must equal the eager
calls bit for bit."""
import pytest
import torch

from gated_delta_rule_46_gb300 import chunk_prefill, decode_step, decode_tokens, inputs
from gpu_util import need_gpu, to_device

pytestmark = pytest.mark.gpu


def _decode_inputs(N, H, d, seed, dev):
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    nrm = lambda s: torch.randn(s, generator=g, device=dev)
    return {"q": torch.nn.functional.normalize(nrm((N, H, d)), dim=-1).to(torch.bfloat16),
            "k": torch.nn.functional.normalize(nrm((N, H, d)), dim=-1).to(torch.bfloat16),
            "v": nrm((N, H, d)).to(torch.bfloat16), "z": nrm((N, H, d)).to(torch.bfloat16),
            "beta": torch.sigmoid(nrm((N, H)))}


def test_decode_steps_in_a_graph():
    dev = need_gpu()
    N, H, d, steps = 16, 4, 128, 3
    A = torch.rand((H, d), device=dev) * 2 - 1
    s0 = 0.1 * torch.randn((N, H, d, d), device=dev)
    bufs = [_decode_inputs(N, H, d, 100, dev) for _ in range(steps)]
    outs = [torch.empty((N, H, d), dtype=torch.bfloat16, device=dev) for _ in range(steps)]
    state = s0.clone()

    def body():
        for b, o in zip(bufs, outs):
            decode_step(b["q"], b["k"], b["v"], b["z"], A, b["beta"], state, out=o)

    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        body()
    for rep in range(2):
        new = [_decode_inputs(N, H, d, 200 + 10 * rep + i, dev) for i in range(steps)]
        for b, n in zip(bufs, new):
            for key in b:
                b[key].copy_(n[key])
        start = state.clone()
        graph.replay()
        torch.cuda.synchronize()
        got_out, got_state = [o.clone() for o in outs], state.clone()
        state.copy_(start)            # eager from the same start state
        body()
        torch.cuda.synchronize()
        for a, b in zip(got_out, outs):
            assert torch.equal(a, b)
        assert torch.equal(got_state, state)


def test_decode_tokens_in_a_graph():
    dev = need_gpu()
    N, n, H, d, P = 12, 4, 2, 128, 20
    A = torch.rand((H, d), device=dev) * 2 - 1
    pool = 0.1 * torch.randn((P, H, d, d), device=dev)
    slots = torch.tensor([5, 0, 19, -1, 7, 3, 11, 2, 14, 9, 1, 16], dtype=torch.int32, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(300)
    nrm = lambda shape: torch.randn(shape, generator=g, device=dev)
    x = {"q": torch.nn.functional.normalize(nrm((N, n, H, d)), dim=-1).to(torch.bfloat16),
         "k": torch.nn.functional.normalize(nrm((N, n, H, d)), dim=-1).to(torch.bfloat16),
         "v": nrm((N, n, H, d)).to(torch.bfloat16), "z": nrm((N, n, H, d)).to(torch.bfloat16),
         "beta": torch.sigmoid(nrm((N, n, H)))}
    out = torch.empty((N, n, H, d), dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        decode_tokens(x["q"], x["k"], x["v"], x["z"], A, x["beta"], pool, slot_ids=slots, out=out)
    start = pool.clone()
    graph.replay()
    torch.cuda.synchronize()
    got_out, got_pool = out.clone(), pool.clone()
    pool.copy_(start)
    decode_tokens(x["q"], x["k"], x["v"], x["z"], A, x["beta"], pool, slot_ids=slots, out=out)
    torch.cuda.synchronize()
    assert torch.equal(got_out, out) and torch.equal(got_pool, pool)


def _plan_sizes(T, N, H):
    from test_gpu_prefill import _plan_workspaces
    return dict(zip(("fused", "windows", "scan"), _plan_workspaces(T, N, H)))


@pytest.mark.parametrize("plan", ["fused", "windows", "scan"])
def test_prefill_plans_in_a_graph(plan):
    dev = need_gpu()
    w = inputs.custom([1500, 33, 900, 640], H=4, dk=128, dv=128, dtype=torch.bfloat16,
                      init="randn0.1", wid=51)
    g = to_device(inputs.prefill_inputs(w), dev)
    T, H = w.total_tokens, w.H
    N = len(w.seq_lens)
    ws = torch.zeros(_plan_sizes(T, N, H)[plan], dtype=torch.uint8, device=dev)
    out = torch.empty((T, H, 128), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((N, H, 128, 128), dtype=torch.float32, device=dev)
    args = (g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"], g["cu_seqlens"], g["initial_state"])
    chunk_prefill(*args, final_state=fin, out=out, workspace=ws)   # first call outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        chunk_prefill(*args, final_state=fin, out=out, workspace=ws)
    d2 = to_device(inputs.prefill_inputs(w, seed=7), dev)          # new inputs, same buffers
    for key in ("q", "k", "v", "z", "beta"):
        g[key].copy_(d2[key])
    graph.replay()
    torch.cuda.synchronize()
    got_out, got_fin = out.clone(), fin.clone()
    chunk_prefill(*args, final_state=fin, out=out, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(got_out, out) and torch.equal(got_fin, fin)
