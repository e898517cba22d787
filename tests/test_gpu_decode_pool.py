"""kda_decode_tokens (several tokens per sequence, states in a slot-indexed
pool) against the oracle, against repeated kda_decode_step calls, and its
handling of padding rows and bad slot ids."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_46_gb300 import KDAError, decode_step, decode_tokens, inputs, kda
from gpu_util import assert_close, need_gpu

pytestmark = pytest.mark.gpu


def _batch(N, n, H, dk, dv, dtype, wid):
    """N sequences of n new tokens each, as [N, n, H, d] tensors (seeded)."""
    w = inputs.custom([n] * N, H=H, dk=dk, dv=dv, dtype=dtype, wid=wid)
    d = inputs.prefill_inputs(w)
    shp = lambda t, last: t.reshape(N, n, H, last)
    return {"q": shp(d["q"], dk), "k": shp(d["k"], dk), "v": shp(d["v"], dv), "z": shp(d["z"], dk),
            "beta": d["beta"].reshape(N, n, H), "A": d["A"], "flat": d, "cu": d["cu_seqlens"]}


@pytest.mark.parametrize("dtype,dk,dv", [(torch.bfloat16, 128, 128), (torch.float32, 64, 32)])
def test_pool_slots_multi_token_against_oracle(dtype, dk, dv):
    dev = need_gpu()
    N, n, H, P = 6, 5, 3, 9
    slots = [3, 7, -1, 0, 8, 5]                   # one padding row; slots 1, 2, 4, 6 untouched
    b = _batch(N, n, H, dk, dv, dtype, wid=41)
    rng = np.random.default_rng(41)
    pool = torch.from_numpy((0.1 * rng.standard_normal((P, H, dk, dv))).astype(np.float32))
    pool_dev = pool.to(dev)
    out = decode_tokens(*(b[x].to(dev) for x in ("q", "k", "v", "z", "A", "beta")), pool_dev,
                        slot_ids=torch.tensor(slots, dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    # the oracle: each row's n tokens as one sequence, starting from its slot's state
    init = np.stack([pool[max(s, 0)].double().numpy() for s in slots])
    f = b["flat"]
    ro, rf = oracle.prefill(f["q"], f["k"], f["v"], f["z"], f["A"], f["beta"], f["cu_seqlens"], init)
    ro = ro.reshape(N, n, H, dv)
    live = [i for i, s in enumerate(slots) if s >= 0]
    assert_close("outputs", out[live], ro[live], dtype)
    assert torch.count_nonzero(out[2]) == 0                      # padding row
    got = pool_dev.cpu()
    assert_close("states", got[[slots[i] for i in live]], rf[live], dtype)
    for s in (1, 2, 4, 6):
        assert torch.equal(got[s], pool[s]), s                   # untouched slots


def test_tokens_equal_repeated_decode_steps():
    """One call over 12 tokens equals 12 kda_decode_step calls (float32)."""
    dev = need_gpu()
    N, n, H, d = 8, 12, 2, 64
    b = _batch(N, n, H, d, d, torch.float32, wid=42)
    rng = np.random.default_rng(42)
    s0 = torch.from_numpy((0.1 * rng.standard_normal((N, H, d, d))).astype(np.float32)).to(dev)
    g = {x: b[x].to(dev) for x in ("q", "k", "v", "z", "A", "beta")}
    pool = s0.clone()
    out = decode_tokens(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"], pool)
    state = s0.clone()
    steps = [decode_step(g["q"][:, t].contiguous(), g["k"][:, t].contiguous(), g["v"][:, t].contiguous(),
                         g["z"][:, t].contiguous(), g["A"], g["beta"][:, t].contiguous(), state)
             for t in range(n)]
    torch.cuda.synchronize()
    ref = torch.stack(steps, dim=1)
    assert torch.allclose(out, ref, rtol=1e-5, atol=1e-6)
    assert torch.allclose(pool, state, rtol=1e-5, atol=1e-6)


def test_bad_slot_is_recorded_and_skipped():
    dev = need_gpu()
    N, n, H, d, P = 3, 2, 2, 32, 4
    b = _batch(N, n, H, d, d, torch.float32, wid=43)
    pool = torch.ones((P, H, d, d), dtype=torch.float32, device=dev)
    status = torch.zeros(256, dtype=torch.uint8, device=dev)
    out = decode_tokens(*(b[x].to(dev) for x in ("q", "k", "v", "z", "A", "beta")), pool,
                        slot_ids=torch.tensor([0, 9, 2], dtype=torch.int32, device=dev), status=status)
    assert kda.check_device_status(status) == kda.KDA_ERR_INVALID_ARG
    assert torch.count_nonzero(out[1]) == 0
    assert torch.equal(pool[1], torch.ones_like(pool[1])) and torch.equal(pool[3], torch.ones_like(pool[3]))
    assert not torch.equal(pool[0], torch.ones_like(pool[0]))


def test_tensor_core_path_two_chunks_and_bad_slot():
    """bf16 128 x 128 heads with several tokens per sequence run the chunked
    form on the tensor cores: 40 tokens (a full and a ragged 32-token chunk)
    per sequence against the oracle, a padding row and a bad slot (recorded,
    padded, no state touched)."""
    dev = need_gpu()
    N, n, H, P = 5, 40, 2, 6
    slots = [4, 9, 0, -1, 2]
    b = _batch(N, n, H, 128, 128, torch.bfloat16, wid=45)
    rng = np.random.default_rng(45)
    pool = torch.from_numpy((0.1 * rng.standard_normal((P, H, 128, 128))).astype(np.float32))
    pool_dev = pool.to(dev)
    status = torch.zeros(256, dtype=torch.uint8, device=dev)
    out = decode_tokens(*(b[x].to(dev) for x in ("q", "k", "v", "z", "A", "beta")), pool_dev,
                        slot_ids=torch.tensor(slots, dtype=torch.int32, device=dev), status=status)
    assert kda.check_device_status(status) == kda.KDA_ERR_INVALID_ARG
    init = np.stack([pool[s].double().numpy() if 0 <= s < P else np.zeros((H, 128, 128)) for s in slots])
    f = b["flat"]
    ro, rf = oracle.prefill(f["q"], f["k"], f["v"], f["z"], f["A"], f["beta"], f["cu_seqlens"], init)
    ro = ro.reshape(N, n, H, 128)
    live = [0, 2, 4]
    assert_close("outputs", out[live], ro[live], torch.bfloat16)
    assert torch.count_nonzero(out[1]) == 0 and torch.count_nonzero(out[3]) == 0
    got = pool_dev.cpu()
    assert_close("states", got[[slots[i] for i in live]], rf[live], torch.bfloat16)
    for s_ in (1, 3, 5):
        assert torch.equal(got[s_], pool[s_]), s_


@pytest.mark.parametrize("n", [4, 8, 13, 32, 33, 40, 45])
def test_tensor_core_path_many_chains_per_cta(n):
    """768 (sequence, head) chains, more than the persistent grid's 2 x SMs
    CTAs, so every CTA runs several chains in a row and fetches the next
    chain's start state and inputs during its current chain's last chunk.
    Padding rows and a bad slot sit where some chains' successors land.
    Last chunks of 4, 8 and 13 valid rows (one 16-token tile, one or two 8-row
    groups), a full 32-row chunk and a 1-row tail. Outputs and states against
    the oracle."""
    dev = need_gpu()
    N, H, P = 96, 8, 112
    rng = np.random.default_rng(46 + n)
    slots = [int(s) for s in rng.permutation(P)[:N]]
    for i in (10, 50, 95):
        slots[i] = -1
    slots[61] = P + 5
    b = _batch(N, n, H, 128, 128, torch.bfloat16, wid=46 + n)
    pool = torch.from_numpy((0.1 * rng.standard_normal((P, H, 128, 128))).astype(np.float32))
    pool_dev = pool.to(dev)
    status = torch.zeros(256, dtype=torch.uint8, device=dev)
    out = decode_tokens(*(b[x].to(dev) for x in ("q", "k", "v", "z", "A", "beta")), pool_dev,
                        slot_ids=torch.tensor(slots, dtype=torch.int32, device=dev), status=status)
    assert kda.check_device_status(status) == kda.KDA_ERR_INVALID_ARG
    init = np.stack([pool[s].double().numpy() if 0 <= s < P else np.zeros((H, 128, 128)) for s in slots])
    f = b["flat"]
    ro, rf = oracle.prefill(f["q"], f["k"], f["v"], f["z"], f["A"], f["beta"], f["cu_seqlens"], init)
    ro = ro.reshape(N, n, H, 128)
    live = [i for i, s in enumerate(slots) if 0 <= s < P]
    assert_close("outputs", out[live], ro[live], torch.bfloat16)
    for i in (10, 50, 61, 95):
        assert torch.count_nonzero(out[i]) == 0, i
    got = pool_dev.cpu()
    assert_close("states", got[[slots[i] for i in live]], rf[live], torch.bfloat16)
    for s_ in sorted(set(range(P)) - {slots[i] for i in live}):
        assert torch.equal(got[s_], pool[s_]), s_


def test_invalid_arguments():
    dev = need_gpu()
    b = _batch(2, 1, 1, 32, 32, torch.float32, wid=44)
    g = [b[x].to(dev) for x in ("q", "k", "v", "z", "A", "beta")]
    small = torch.zeros((1, 1, 32, 32), dtype=torch.float32, device=dev)
    with pytest.raises(KDAError):          # no slot ids and a pool smaller than N
        decode_tokens(*g, small)


def test_prefill_to_decode_handoff_through_pool():
    """Prefill N prompts, move the final states into pool slots, then decode n
    more tokens per sequence from the pool: outputs and states equal the
    oracle over the whole sequences."""
    from gated_delta_rule_46_gb300 import chunk_prefill, state_slots_copy
    dev = need_gpu()
    lens, n, H, d, P = [70, 1, 130, 64, 9], 4, 2, 128, 11
    slots = [7, 2, 10, 0, 5]
    N = len(lens)
    w = inputs.custom([L + n for L in lens], H=H, dk=d, dv=d, dtype=torch.bfloat16, init="randn0.1", wid=45)
    f = inputs.prefill_inputs(w)
    cu = f["cu_seqlens"].tolist()
    pre = torch.cat([torch.arange(cu[i], cu[i] + lens[i]) for i in range(N)])
    new = torch.cat([torch.arange(cu[i] + lens[i], cu[i + 1]) for i in range(N)])
    cu_pre = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    g = {x: f[x].to(dev) for x in ("q", "k", "v", "z", "beta")}
    A = f["A"].to(dev)
    _, fin = chunk_prefill(*(g[x][pre.to(dev)].contiguous() for x in ("q", "k", "v", "z")), A,
                           g["beta"][pre.to(dev)].contiguous(), cu_pre.to(dev), f["initial_state"].to(dev))
    pool = torch.full((P, H, d, d), 3.0, dtype=torch.float32, device=dev)
    sl = torch.tensor(slots, dtype=torch.int32, device=dev)
    state_slots_copy(pool, sl, fin, to_pool=True)
    shp = lambda t, last: t[new.to(dev)].reshape(N, n, H, last).contiguous()
    out = decode_tokens(shp(g["q"], d), shp(g["k"], d), shp(g["v"], d), shp(g["z"], d), A,
                        g["beta"][new.to(dev)].reshape(N, n, H).contiguous(), pool, slot_ids=sl)
    back = state_slots_copy(pool, torch.tensor([0, -1, 7], dtype=torch.int32, device=dev),
                            torch.full((3, H, d, d), 5.0, dtype=torch.float32, device=dev), to_pool=False)
    torch.cuda.synchronize()
    ro, rf = oracle.prefill(f["q"], f["k"], f["v"], f["z"], f["A"], f["beta"], f["cu_seqlens"], f["initial_state"])
    assert_close("outputs", out.reshape(-1, H, d), ro[new.numpy()], torch.bfloat16)
    assert_close("states", pool[sl.long()], rf, torch.bfloat16)
    for s_ in range(P):
        if s_ not in slots:
            assert torch.all(pool[s_] == 3.0), s_          # untouched slots
    assert torch.equal(back[0], pool[0]) and torch.equal(back[2], pool[7])
    assert torch.count_nonzero(back[1]) == 0               # padding row zeroed
