"""Pins for the fp64 CPU oracle (``oracle/``), run on the CPU only.

The oracle is the yardstick for every GPU parity test, so it is checked here
against things other than itself:

* gate: exact rational values from ``golden/gate_special_values.txt``
  (hand-derived from the printed gate formula), the identity
  g(z) + g(-z) = g_min, scipy's logistic function, and the saturation limits;
* the bound the pages state: every gate value in (-5, 0) and every 16-token
  window of cumulative log-decay in (-80, 0) on the benchmark inputs;
* closed forms of the recurrence that do not use its update formula:
  beta = 0 gives pure channel-wise decay; alpha = 1, beta = 1 and orthonormal
  keys give exact key -> value retrieval; beta = 1 with unit keys makes the
  state return v_t for k_t right after the write (the delta rule's defining
  property);
* two independently derived formulations: the generalised-Householder product
  form with explicit dense matrices, and the chunkwise WY/UT form (the algebra
  the GPU kernels implement) for chunk sizes 1, 4, 16 and 64 with ragged tails;
* the affine segment maps behind the GPU's segment scan: the chunk-formula
  transition M equals the map the oracle realises, and composing segments
  with S_in(g+1) = M_g S_in(g) + S0_g reproduces a single call;
* structural properties: packed sequences are independent, a split resumed
  from the carried state equals one call, T decode steps equal a T-token
  prefill, and the norm bound ||S_t|| <= ||S_{t-1}|| + beta ||v_t||;
* a mutation check: plausible mistakes planted in a copy of the oracle's C
  source (dropped decay, decay after the write, wrong sign, missing beta,
  transposed read, q/k swapped, wrong gate sign) each fail at least one pin.
"""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import scipy.special

import oracle
from gated_delta_rule_46_gb300 import inputs

HERE = os.path.dirname(os.path.abspath(__file__))
G_MIN = -5.0


def _rand_problem(rng, lens, H, dk, dv, unit_keys=True, init=True):
    T = int(sum(lens))
    q = rng.standard_normal((T, H, dk)).astype(np.float32)
    k = rng.standard_normal((T, H, dk)).astype(np.float32)
    if unit_keys:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv)).astype(np.float32)
    z = rng.standard_normal((T, H, dk)).astype(np.float32)
    A = rng.uniform(-1, 1, (H, dk)).astype(np.float32)
    beta = (1 / (1 + np.exp(-rng.standard_normal((T, H))))).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    s0 = (0.1 * rng.standard_normal((len(lens), H, dk, dv))) if init else None
    return dict(q=q, k=k, v=v, z=z, A=A, beta=beta, cu=cu, s0=s0)


def _run(p, g=None, **kw):
    return oracle.prefill(p["q"], p["k"], p["v"], p["z"], p["A"], p["beta"], p["cu"],
                          initial_state=p["s0"], g=g, **kw)


# --------------------------------------------------------------------------- gate

def test_gate_golden_values():
    rows = []
    with open(os.path.join(HERE, "golden", "gate_special_values.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    rows = np.array(rows)
    z = rows[:, 0].astype(np.float32).reshape(-1, 1, 1)
    for i in range(len(rows)):
        A = np.full((1, 1), rows[i, 1], dtype=np.float32)
        g = oracle.gate(z[i:i + 1], A)[0, 0, 0]
        assert abs(g - rows[i, 2]) < 2e-6, (rows[i], g)


def test_gate_symmetry_scipy_and_limits():
    rng = np.random.default_rng(1)
    z = rng.standard_normal((50, 3, 16)).astype(np.float32) * 3
    A = rng.uniform(-1, 1, (3, 16)).astype(np.float32)
    g = oracle.gate(z, A)
    gm = oracle.gate(-z, A)
    # sigmoid(x) + sigmoid(-x) = 1  =>  g(z) + g(-z) = g_min
    assert np.max(np.abs(g + gm - G_MIN)) < 1e-13
    x = np.exp(A.astype(np.float64))[None] * z.astype(np.float64)
    ref = G_MIN * scipy.special.expit(x)
    assert np.max(np.abs(g - ref)) < 1e-13
    assert np.all(g < 0) and np.all(g > G_MIN)
    big = oracle.gate(np.array([[[40.0, -40.0, 0.0]]], np.float32), np.zeros((1, 3), np.float32))
    assert abs(big[0, 0, 0] - G_MIN) < 1e-15
    assert -1e-16 < big[0, 0, 1] < 0
    assert big[0, 0, 2] == -2.5


@pytest.mark.parametrize("wid", [0, 1, 4])
def test_gate_bound_on_workloads(wid):
    """Every gate value lies in (-5, 0) and every 16-token window of cumulative
    log-decay lies in (-80, 0) (the tile bound stated for the gate floor)."""
    w = inputs.workload(wid)
    if w.decode_N:
        z = inputs.decode_inputs(w, 0)["z"]
        A = inputs.decode_A(w)
    else:
        d = inputs.prefill_inputs(w)
        z, A = d["z"], d["A"]
    g = oracle.gate(z, A)
    assert np.all(g < 0) and np.all(g > G_MIN)
    if not w.decode_N:
        c = np.cumsum(g, axis=0)
        c = np.concatenate([np.zeros_like(c[:1]), c], axis=0)
        win = c[16:] - c[:-16]
        assert np.all(win < 0) and np.all(win > 16 * G_MIN)


def test_gate_bound_on_large_workload_slab():
    w = inputs.workload(3)
    d = inputs.prefill_inputs(w, t0=0, t1=2048)
    g = oracle.gate(d["z"], d["A"])
    c = np.concatenate([np.zeros_like(g[:1]), np.cumsum(g, axis=0)], axis=0)
    win = c[16:] - c[:-16]
    assert np.all(g > G_MIN) and np.all(g < 0)
    assert np.all(win > -80) and np.all(win < 0)


# --------------------------------------------------------------------------- closed forms

def test_beta_zero_is_pure_channel_decay():
    rng = np.random.default_rng(2)
    p = _rand_problem(rng, [7, 5], 2, 6, 4)
    p["beta"][:] = 0
    out, fin = _run(p)
    g = oracle.gate(p["z"], p["A"])
    for i in range(2):
        b, e = p["cu"][i], p["cu"][i + 1]
        for h in range(2):
            G = np.cumsum(g[b:e, h], axis=0)          # [n, dk]
            S0 = p["s0"][i, h]
            for t in range(e - b):
                St = np.exp(G[t])[:, None] * S0
                np.testing.assert_allclose(out[b + t, h], St.T @ p["q"][b + t, h], rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(fin[i, h], np.exp(G[-1])[:, None] * S0, rtol=1e-12, atol=1e-14)


def test_unit_decay_orthonormal_keys_retrieve_values():
    rng = np.random.default_rng(3)
    dk, dv, n = 8, 5, 6
    Q, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Q[:n].astype(np.float32)                # orthonormal rows
    p = _rand_problem(rng, [n], 1, dk, dv, init=False)
    p["k"][:, 0] = keys
    p["q"][:, 0] = keys[0]                          # always ask for the first key
    p["beta"][:] = 1
    g = np.zeros((n, 1, dk))
    out, fin = _run(p, g=g)
    V = p["v"][:, 0].astype(np.float64)
    K = keys.astype(np.float64)
    # keys are only float32-orthonormal: tolerance from their rounding
    np.testing.assert_allclose(fin[0, 0], K.T @ V, atol=1e-6)
    for t in range(n):
        np.testing.assert_allclose(out[t, 0], V[0], atol=1e-6)


def test_delta_rule_write_returns_value():
    """beta = 1 and ||k_t|| = 1: right after the write, S_t^T k_t = v_t for any decay."""
    rng = np.random.default_rng(4)
    p = _rand_problem(rng, [9, 4], 2, 8, 3)
    k64 = p["k"].astype(np.float64)
    p["k"] = (k64 / np.linalg.norm(k64, axis=-1, keepdims=True)).astype(np.float32)
    p["q"] = p["k"].copy()
    p["beta"][:] = 1
    out, _ = _run(p)
    nk = np.linalg.norm(p["k"].astype(np.float64), axis=-1)
    # o_t = S_t^T k_t = v_t + (1 - ||k||^2) * (...) ; float32 keys have ||k||^2 = 1 +- 1e-7
    np.testing.assert_allclose(out, p["v"].astype(np.float64), atol=5e-6)
    assert np.max(np.abs(nk - 1)) < 1e-6


# --------------------------------------------------------------------------- other formulations

def _householder_form(p, g):
    """S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T, dense matrices."""
    q, k, v, beta, cu = (p[n].astype(np.float64) if n != "cu" else p[n]
                         for n in ("q", "k", "v", "beta", "cu"))
    T, H, dk = q.shape
    dv = v.shape[2]
    out = np.zeros((T, H, dv))
    fin = np.zeros((len(cu) - 1, H, dk, dv))
    for i in range(len(cu) - 1):
        for h in range(H):
            S = np.zeros((dk, dv)) if p["s0"] is None else p["s0"][i, h].copy()
            for t in range(cu[i], cu[i + 1]):
                kt = k[t, h][:, None]
                M = (np.eye(dk) - beta[t, h] * kt @ kt.T) @ np.diag(np.exp(g[t, h]))
                S = M @ S + beta[t, h] * kt @ v[t, h][None, :]
                out[t, h] = S.T @ q[t, h]
            fin[i, h] = S
    return out, fin


def _chunked_form(p, g, C):
    """Chunkwise WY/UT form: within a chunk with start state S0 and inclusive
    cumulative log-decay G,  (I + L) U = Diag(beta)(V - K~ S0),
    L_ts = beta_t sum_c k_tc k_sc e^{G_tc - G_sc} (s < t),  O = Q~ S0 + P U,
    P_ts = sum_c q_tc k_sc e^{G_tc - G_sc} (s <= t),
    S_end = Diag(e^{G_end}) S0 + (K * e^{G_end - G})^T U."""
    q, k, v, beta = (p[n].astype(np.float64) for n in ("q", "k", "v", "beta"))
    cu = p["cu"]
    T, H, dk = q.shape
    dv = v.shape[2]
    out = np.zeros((T, H, dv))
    fin = np.zeros((len(cu) - 1, H, dk, dv))
    for i in range(len(cu) - 1):
        for h in range(H):
            S = np.zeros((dk, dv)) if p["s0"] is None else p["s0"][i, h].copy()
            for c0 in range(cu[i], cu[i + 1], C):
                c1 = min(c0 + C, cu[i + 1])
                n = c1 - c0
                K, Q, V, b = k[c0:c1, h], q[c0:c1, h], v[c0:c1, h], beta[c0:c1, h]
                G = np.cumsum(g[c0:c1, h], axis=0)
                diff = G[:, None, :] - G[None, :, :]                 # [t, s, c]
                causal = np.tril(np.ones((n, n), bool))[:, :, None]
                D = np.exp(np.where(causal, diff, -np.inf))
                Akk = np.einsum("tc,sc,tsc->ts", K, K, D)
                L = np.tril(Akk, -1) * b[:, None]
                Tm = np.linalg.solve(np.eye(n) + L, np.diag(b))
                Kt, Qt = K * np.exp(G), Q * np.exp(G)
                U = Tm @ V - (Tm @ Kt) @ S
                P = np.einsum("tc,sc,tsc->ts", Q, K, D)
                out[c0:c1, h] = Qt @ S + P @ U
                Kend = K * np.exp(G[-1][None, :] - G)
                S = np.exp(G[-1])[:, None] * S + Kend.T @ U
            fin[i, h] = S
    return out, fin


def test_householder_product_form_matches():
    rng = np.random.default_rng(5)
    p = _rand_problem(rng, [11, 1, 6], 2, 5, 3)
    out, fin = _run(p)
    g = oracle.gate(p["z"], p["A"])
    ho, hf = _householder_form(p, g)
    np.testing.assert_allclose(out, ho, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(fin, hf, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("C", [1, 4, 7, 16, 32, 64])   # 16, 32, 64: the chunk sizes of the GPU kernels
def test_chunked_wy_form_matches(C):
    rng = np.random.default_rng(6 + C)
    p = _rand_problem(rng, [70, 17, 1, 33], 2, 8, 6)
    out, fin = _run(p)
    g = oracle.gate(p["z"], p["A"])
    co, cf = _chunked_form(p, g, C)
    scale = np.max(np.abs(out))
    assert np.max(np.abs(out - co)) <= 1e-10 * scale
    assert np.max(np.abs(fin - cf)) <= 1e-10 * np.max(np.abs(fin))


def test_chunked_wy_form_unit_decay_and_zero_state():
    rng = np.random.default_rng(7)
    p = _rand_problem(rng, [40], 1, 4, 4, init=False)
    g = np.zeros((40, 1, 4))
    out, fin = _run(p, g=g)
    co, cf = _chunked_form(p, g, 16)
    np.testing.assert_allclose(out, co, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(fin, cf, rtol=1e-10, atol=1e-12)


def _segment_map(p, g, h, t0, t1, C):
    """Transition of the state over tokens [t0, t1) (whole chunks of C from t0),
    by the chunk formula the GPU's segment pass propagates:
    M = prod_chunks (Diag(e^{G_end}) - Kend^T T K~), later chunks on the left."""
    k, beta = p["k"].astype(np.float64), p["beta"].astype(np.float64)
    dk = k.shape[2]
    M = np.eye(dk)
    for c0 in range(t0, t1, C):
        c1 = min(c0 + C, t1)
        n = c1 - c0
        K, b = k[c0:c1, h], beta[c0:c1, h]
        G = np.cumsum(g[c0:c1, h], axis=0)
        diff = G[:, None, :] - G[None, :, :]
        D = np.exp(np.where(np.tril(np.ones((n, n), bool))[:, :, None], diff, -np.inf))
        L = np.tril(np.einsum("tc,sc,tsc->ts", K, K, D), -1) * b[:, None]
        Tm = np.linalg.solve(np.eye(n) + L, np.diag(b))
        W = Tm @ (K * np.exp(G))
        Kend = K * np.exp(G[-1][None, :] - G)
        M = (np.diag(np.exp(G[-1])) - Kend.T @ W) @ M
    return M


def test_segment_maps_compose_affinely():
    """The state map over a segment is affine, S_out = M S_in + S0, with M the
    chunk-formula product above and S0 the segment run from a zero state; the
    scan S_in(g+1) = M_g S_in(g) + S0_g over three segments reproduces the
    whole sequence's final state and, resumed from S_in(g), its outputs.  Slow
    decay (g near 0) and small beta keep M far from 0 so every term matters."""
    rng = np.random.default_rng(11)
    dk = dv = 6
    lens, H, C = [96], 1, 16
    p = _rand_problem(rng, lens, H, dk, dv)
    p["beta"] = (0.05 * p["beta"]).astype(np.float32)   # gentle writes: the delta rule forgets slowly too
    g = -0.02 * np.abs(rng.standard_normal((96, H, dk)))
    out, fin = _run(p, g=g)
    S = p["s0"][0, 0].copy()
    for t0, t1 in [(0, 32), (32, 80), (80, 96)]:
        sub = {n: (p[n][t0:t1] if n in ("q", "k", "v", "z", "beta") else p[n]) for n in p}
        sub["cu"] = np.array([0, t1 - t0], dtype=np.int64)
        gs = g[t0:t1]
        M = _segment_map(p, g, 0, t0, t1, C)
        assert np.abs(M).max() > 0.2                                  # far from decayed away
        sub["s0"] = np.zeros((1, H, dk, dv))
        _, S0 = _run(sub, g=gs)
        sub["s0"] = np.eye(dk)[None, None]                            # dv = dk: S_in = I gives M + S0
        _, SI = _run(sub, g=gs)
        np.testing.assert_allclose(SI[0, 0] - S0[0, 0], M, rtol=1e-9, atol=1e-11)
        sub["s0"] = S[None, None]
        seg_out, seg_fin = _run(sub, g=gs)
        np.testing.assert_allclose(seg_out, out[t0:t1], rtol=1e-9, atol=1e-11)
        S = M @ S + S0[0, 0]                                          # the scan step
        np.testing.assert_allclose(seg_fin[0, 0], S, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(S, fin[0, 0], rtol=1e-9, atol=1e-11)


# --------------------------------------------------------------------------- structure

def test_packed_sequences_are_independent():
    rng = np.random.default_rng(8)
    p = _rand_problem(rng, [5, 0, 9, 3], 2, 4, 3)
    out, fin = _run(p)
    for i in range(4):
        b, e = p["cu"][i], p["cu"][i + 1]
        sub = {n: p[n][b:e] for n in ("q", "k", "v", "z", "beta")}
        sub.update(A=p["A"], cu=np.array([0, e - b]), s0=p["s0"][i:i + 1])
        o1, f1 = _run(sub)
        assert np.array_equal(o1, out[b:e]) and np.array_equal(f1[0], fin[i])
    assert np.array_equal(fin[1], p["s0"][1])      # empty sequence: state passes through


def test_split_and_resume_equals_single_call():
    rng = np.random.default_rng(9)
    p = _rand_problem(rng, [29], 2, 6, 5)
    out, fin = _run(p)
    for cut in (1, 13, 28):
        a = {n: p[n][:cut] for n in ("q", "k", "v", "z", "beta")}
        a.update(A=p["A"], cu=np.array([0, cut]), s0=p["s0"])
        oa, fa = _run(a)
        b = {n: p[n][cut:] for n in ("q", "k", "v", "z", "beta")}
        b.update(A=p["A"], cu=np.array([0, 29 - cut]), s0=fa)
        ob, fb = _run(b)
        assert np.array_equal(np.concatenate([oa, ob]), out) and np.array_equal(fb, fin)


def test_decode_steps_equal_prefill():
    rng = np.random.default_rng(10)
    N, H, dk, dv, T = 3, 2, 5, 4, 6
    lens = [T] * N
    p = _rand_problem(rng, lens, H, dk, dv)
    out, fin = _run(p)
    st = p["s0"].copy()
    for t in range(T):
        idx = [i * T + t for i in range(N)]
        o, st = oracle.decode_step(p["q"][idx], p["k"][idx], p["v"][idx], p["z"][idx],
                                   p["A"], p["beta"][idx], st)
        assert np.array_equal(o, out[idx])
    assert np.array_equal(st, fin)


def test_state_norm_bound():
    rng = np.random.default_rng(11)
    p = _rand_problem(rng, [24], 1, 6, 4)
    prev = np.linalg.norm(p["s0"][0, 0], 2)
    for t in range(1, 25):
        sub = {n: p[n][:t] for n in ("q", "k", "v", "z", "beta")}
        sub.update(A=p["A"], cu=np.array([0, t]), s0=p["s0"])
        _, f = _run(sub)
        cur = np.linalg.norm(f[0, 0], 2)
        vb = p["beta"][t - 1, 0] * np.linalg.norm(p["v"][t - 1, 0].astype(np.float64))
        assert cur <= prev + vb + 1e-12
        prev = cur


def test_rejects_bad_arguments():
    rng = np.random.default_rng(12)
    p = _rand_problem(rng, [4], 1, 4, 4)
    p["cu"] = np.array([3, 1], dtype=np.int64)                       # decreasing offsets
    with pytest.raises(ValueError):
        _run(p)


# --------------------------------------------------------------------------- mutations

_MUTANTS = {
    "dropped_decay": ("S[(int64_t)c * dv + j] *= alpha[c];", ";"),
    "decay_after_write": (
        "S[(int64_t)c * dv + j] *= alpha[c];", ";",
        "for (int j = 0; j < dv; ++j) S[(int64_t)c * dv + j] += kc * u[j];",
        "for (int j = 0; j < dv; ++j) S[(int64_t)c * dv + j] = (S[(int64_t)c * dv + j] + kc * u[j]) * alpha[c];"),
    "wrong_sign_u": ("u[j] = b * ((double)job->v[rv + j] - kv[j]);",
                     "u[j] = b * ((double)job->v[rv + j] + kv[j]);"),
    "missing_beta": ("u[j] = b * ((double)job->v[rv + j] - kv[j]);",
                     "u[j] = ((double)job->v[rv + j] - kv[j]);"),
    "transposed_read": ("kv[j] += S[(int64_t)c * dv + j] * kc;",
                        "kv[j] += S[(int64_t)(j % dk) * dv + (c % dv)] * kc;"),
    "q_for_k_in_read": ("double kc = (double)job->k[rk + c];\n            for (int j = 0; j < dv; ++j) kv[j]",
                        "double kc = (double)job->q[rk + c];\n            for (int j = 0; j < dv; ++j) kv[j]"),
    "gate_sign": ("return KDA_ORACLE_G_MIN / (1.0 + exp(-x));",
                  "return KDA_ORACLE_G_MIN / (1.0 + exp(x));"),
    "gate_no_expA": ("double x = exp(A) * z;", "double x = A * z;"),
    "output_from_pre_write_state": ("o[j] += S[(int64_t)c * dv + j] * qc;",
                                    "o[j] += (S[(int64_t)c * dv + j] - (double)job->k[rk + c] * u[j]) * qc;"),
}


def _pins_pass(mod):
    """The pin checks above, re-run against a (possibly mutated) oracle module."""
    saved = oracle._lib
    try:
        oracle._lib = mod
        checks = [test_gate_golden_values, test_gate_symmetry_scipy_and_limits,
                  test_beta_zero_is_pure_channel_decay,
                  test_unit_decay_orthonormal_keys_retrieve_values,
                  test_delta_rule_write_returns_value, test_householder_product_form_matches,
                  lambda: test_chunked_wy_form_matches(16), test_split_and_resume_equals_single_call,
                  test_packed_sequences_are_independent]
        for chk in checks:
            try:
                with np.errstate(all="ignore"):
                    chk()
            except (AssertionError, ValueError, FloatingPointError):
                return False
        return True
    finally:
        oracle._lib = saved


def test_unmutated_oracle_passes_pins():
    oracle._load()
    assert _pins_pass(oracle._lib)


@pytest.mark.parametrize("name", sorted(_MUTANTS))
def test_planted_mistake_is_caught(name):
    import ctypes
    src = open(oracle._SRC).read()
    edits = _MUTANTS[name]
    for a, b in zip(edits[0::2], edits[1::2]):
        assert a in src, (name, a)
        src = src.replace(a, b, 1)
    d = tempfile.mkdtemp(prefix="kda_mut_")
    try:
        cfile, so = os.path.join(d, "m.c"), os.path.join(d, "m.so")
        open(cfile, "w").write(src)
        subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                        "-pthread", cfile, "-o", so, "-lm"], check=True)
        lib = ctypes.CDLL(so)
        ref = oracle._load()
        for fn in ("kda_oracle_gate", "kda_oracle_prefill", "kda_oracle_decode_step"):
            getattr(lib, fn).argtypes = getattr(ref, fn).argtypes
            getattr(lib, fn).restype = getattr(ref, fn).restype
        assert not _pins_pass(lib), f"mutant {name} survived every pin"
    finally:
        shutil.rmtree(d, ignore_errors=True)
