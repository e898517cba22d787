"""Context parallelism on the GPU: kda_segment_map and kda_state_compose
against the oracle, and the whole driver on two gloo ranks that share cuda:0
(each a process of its own; their kernels never wait on one another, the maps
travel through the host), each holding half of the sequences, against one
oracle pass over the whole sequences."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_46_gb300 import (check_device_status, inputs, segment_map,
                                       segment_map_workspace_size, state_compose)
from cp_util import rank_segments, run_ranks
from gpu_util import assert_close, need_gpu, to_device

pytestmark = pytest.mark.gpu


def _batch(lens, slow, wid):
    w = inputs.custom(lens, H=2, dk=128, dv=128, dtype=torch.bfloat16, init="randn0.1", wid=wid)
    d = inputs.prefill_inputs(w)
    if slow:   # gates near 0: the maps keep memory over the whole segment
        d["z"] = (d["z"].float() - 10.0).to(torch.bfloat16)
    return d


def _oracle_maps(d):
    T, H, dk = d["q"].shape
    N = d["cu_seqlens"].numel() - 1
    _, b = oracle.prefill(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["cu_seqlens"], None)
    eye = np.broadcast_to(np.eye(dk), (N, H, dk, dk)).copy()
    _, M = oracle.prefill(d["q"], d["k"], torch.zeros((T, H, dk)), d["z"], d["A"], d["beta"],
                          d["cu_seqlens"], eye)
    return M, b


@pytest.mark.parametrize("slow", [False, True])
def test_segment_map_matches_oracle(slow):
    """M (the linear part, from the identity with v = 0 in the oracle) and b
    (from a zero state) of every (sequence, head), including an empty sequence
    (M = I, b = 0) and one shorter than a chunk."""
    dev = need_gpu()
    lens = [1500, 900, 0, 37, 4100]
    d = _batch(lens, slow, 71)
    g = to_device(d, dev)
    T, N = sum(lens), len(lens)
    ws = torch.zeros(segment_map_workspace_size(T, N, 2, 128, 128), dtype=torch.uint8, device=dev)
    M, b = segment_map(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"], g["cu_seqlens"], workspace=ws)
    assert check_device_status(ws) == 0
    rM, rb = _oracle_maps(d)
    assert_close("M", M, rM, torch.bfloat16)
    assert_close("b", b, rb, torch.bfloat16)
    assert torch.equal(M[2].cpu(), torch.eye(128).expand(2, 128, 128))
    assert torch.count_nonzero(b[2]) == 0


def test_state_compose_matches_float64():
    dev = need_gpu()
    rng = np.random.default_rng(5)
    R, N, H, dk, dv = 3, 2, 3, 128, 64
    M = rng.standard_normal((R, N, H, dk, dk)) / np.sqrt(dk)
    b = rng.standard_normal((R, N, H, dk, dv))
    s0 = rng.standard_normal((N, H, dk, dv))
    st = state_compose(torch.tensor(M, dtype=torch.float32, device=dev),
                       torch.tensor(b, dtype=torch.float32, device=dev),
                       torch.tensor(s0, dtype=torch.float32, device=dev))
    ref = [s0]
    for r in range(R):
        ref.append(M[r] @ ref[-1] + b[r])
    ref = np.stack(ref)
    got = st.double().cpu().numpy()
    err = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err < 1e-5, err
    st0 = state_compose(torch.empty((0, N, H, dk, dk), device=dev), torch.empty((0, N, H, dk, dv), device=dev))
    assert st0.shape == (1, N, H, dk, dv) and torch.count_nonzero(st0) == 0


def _gpu_rank(rank, world, segs, init):
    import torch
    from gated_delta_rule_46_gb300.context_parallel import context_parallel_prefill
    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    s = {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in segs[rank].items()}
    out, s_out, s_in = context_parallel_prefill(s["q"], s["k"], s["v"], s["z"], s["A"], s["beta"],
                                                s["cu_seqlens"], init.to(dev))
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), s_out.cpu().numpy(), s_in.cpu().numpy()


@pytest.mark.parametrize("slow", [False, True])
def test_two_ranks_on_one_gpu_equal_one_pass(slow):
    need_gpu()
    lens = [3000, 700, 1300]
    cuts = [[1400], [700], [333]]          # rank 1 holds nothing of the second sequence
    d = _batch(lens, slow, 72)
    segs = rank_segments(d, lens, cuts)
    res = run_ranks(2, _gpu_rank, segs, d["initial_state"])
    ro, rf = oracle.prefill(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["cu_seqlens"],
                            d["initial_state"])
    got = np.zeros(ro.shape, dtype=np.float64)
    for r in range(2):
        out = res[r][0]
        pos = 0
        for a, b in segs[r]["spans"]:
            got[a:b] = out[pos:pos + (b - a)]
            pos += b - a
    assert_close("outputs of both ranks", got, ro, torch.bfloat16)
    assert_close("final states (last rank)", res[1][1], rf, torch.bfloat16)
    # rank 1's incoming states equal the oracle's states at the cuts
    cu = np.concatenate([[0], np.cumsum(lens)])
    cut_d = {n: torch.cat([d[n][int(cu[i]):int(cu[i]) + cuts[i][0]] for i in range(len(lens))])
             for n in ("q", "k", "v", "z", "beta")}
    cu_cut = np.concatenate([[0], np.cumsum([c[0] for c in cuts])])
    _, s_mid = oracle.prefill(cut_d["q"], cut_d["k"], cut_d["v"], cut_d["z"], d["A"], cut_d["beta"],
                              cu_cut, d["initial_state"])
    assert_close("incoming state of rank 1", res[1][2], s_mid, torch.bfloat16)
