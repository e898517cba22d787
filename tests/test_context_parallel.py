"""The exchange logic of the context-parallel prefill on CPU gloo ranks.

gated_delta_rule_46_gb300.context_parallel orders four steps on every rank:
the affine map of its segments, one all_gather of the maps, the composition of
the maps of the ranks before it (an exclusive scan) and the rerun of its
segments from the composed incoming state.  Here the three compute steps are
the fp64 oracle, run on world-size-2 and -3 gloo groups of processes: the
segment's map from the oracle (b = the segment from a zero state; M, by
linearity, the segment with v = 0 from the identity), the composition a plain
matrix loop, the rerun the oracle from the given state.  The outputs of all
ranks, put back together, and the last rank's final states must then equal
one oracle pass over the whole sequences; a wrong rank order, an inclusive
instead of exclusive scan or a dropped map all fail that.
"""
import numpy as np
import pytest
import torch

from cp_util import rank_segments, run_ranks


class OracleOps:
    """The compute steps of the driver, done by the oracle in float64."""

    def segment_map(self, q, k, v, z, A, beta, cu_seqlens):
        import oracle
        T, H, dk = q.shape
        N = cu_seqlens.numel() - 1
        _, b = oracle.prefill(q, k, v, z, A, beta, cu_seqlens, None)
        eye = np.broadcast_to(np.eye(dk), (N, H, dk, dk)).copy()
        _, M = oracle.prefill(q, k, torch.zeros((T, H, dk)), z, A, beta, cu_seqlens, eye)
        return torch.from_numpy(M), torch.from_numpy(b)

    def state_compose(self, M, b, initial_state):
        s = torch.zeros(b.shape[1:], dtype=torch.float64) if initial_state is None else initial_state
        states = [s]
        for r in range(M.shape[0]):
            s = M[r] @ s + b[r]
            states.append(s)
        return torch.stack(states)

    def chunk_prefill(self, q, k, v, z, A, beta, cu_seqlens, initial_state):
        import oracle
        out, fin = oracle.prefill(q, k, v, z, A, beta, cu_seqlens, initial_state.numpy())
        return torch.from_numpy(out), torch.from_numpy(fin)


def _rank_fn(rank, world, segs, init):
    from gated_delta_rule_46_gb300.context_parallel import context_parallel_prefill
    s = segs[rank]
    out, s_out, s_in = context_parallel_prefill(s["q"], s["k"], s["v"], s["z"], s["A"], s["beta"],
                                                s["cu_seqlens"], init, ops=OracleOps())
    return out.numpy(), s_out.numpy(), s_in.numpy()


@pytest.mark.parametrize("world,lens,cuts", [
    (2, [150, 97], [[64], [97]]),            # rank 1 holds nothing of the second sequence
    (3, [200, 61, 130], [[1, 90], [30, 30], [0, 129]]),   # empty and one-token segments
])
def test_context_parallel_equals_one_pass(world, lens, cuts):
    import oracle
    from gated_delta_rule_46_gb300 import inputs
    w = inputs.custom(lens, H=2, dk=32, dv=32, dtype=torch.float32, init="randn0.1", wid=61)
    d = inputs.prefill_inputs(w)
    init = d["initial_state"].double()
    segs = rank_segments(d, lens, cuts)
    res = run_ranks(world, _rank_fn, segs, init)
    ro, rf = oracle.prefill(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["cu_seqlens"],
                            d["initial_state"])
    got = np.zeros_like(ro)
    for r in range(world):
        out, _, _ = res[r]
        pos = 0
        for a, b in segs[r]["spans"]:
            got[a:b] = out[pos:pos + (b - a)]
            pos += b - a
    np.testing.assert_allclose(got, ro, rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(res[-1][1], rf, rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(res[0][2], init.numpy(), rtol=0, atol=0)   # rank 0 starts from the initial state
