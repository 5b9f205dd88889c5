"""Pins of the fp64 oracle (C token loop and numpy chunk mirror).

CPU only.  The pins come from closed forms, special cases and invariants
(tests/_pins.py), from the constants the pages print (tests/golden/) and
from brute-force agreement of the chunked form with the token loop.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import chunk_mirror
from kda_inputs import WORKLOADS, make_unit
from tests import _pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "paper_constants.txt")


def _golden():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, val, tol = line.split()[:3]
            out[name] = (float(val), float(tol))
    return out


def c_unit(q, k, v, g, beta, s0):
    return oracle.fwd_unit(q, k, v, g, beta, s0)


def mirror_unit(C):
    def f(q, k, v, g, beta, s0):
        return chunk_mirror.forward_unit(q, k, v, g, beta, s0, chunk=C)
    return f


@pytest.mark.parametrize("pin", _pins.ALL, ids=lambda p: p.__name__)
def test_c_oracle_pins(pin):
    ok, err = pin(c_unit)
    assert ok, (pin.__name__, err)


@pytest.mark.parametrize("C", [1, 4, 16, 64])
@pytest.mark.parametrize("pin", _pins.ALL, ids=lambda p: p.__name__)
def test_chunk_mirror_pins(pin, C):
    ok, err = pin(mirror_unit(C))
    if pin is _pins.p1_retrieval or pin is _pins.p2_beta_zero or pin is _pins.p8_affine:
        # the chunked form rounds differently from the token loop; these
        # identities hold to rounding, not bit for bit
        ok = err < 1e-10
    elif pin is _pins.p10_split:
        ok = err < 1e-10
    else:
        ok = ok or err < 1e-10
    assert ok, (pin.__name__, C, err)


# ---- gate: negative softplus with the -5 floor ------------------------------

def test_gate_textbook():
    x = np.concatenate([np.linspace(-40, 40, 2001), [-700.0, -200.0, 0.0, 4.9932, 700.0]])
    a = oracle.log_decay(x)
    ref = np.array([max(-math.log1p(math.exp(t)) if t < 30 else -(t + math.log1p(math.exp(-t))),
                        -5.0) for t in x])
    np.testing.assert_allclose(a, ref, rtol=1e-15, atol=1e-300)
    np.testing.assert_allclose(chunk_mirror.log_decay(x), ref, rtol=1e-15, atol=1e-300)
    assert oracle.log_decay(np.array([0.0]))[0] == pytest.approx(-math.log(2.0), rel=1e-15)
    assert oracle.log_decay(np.array([50.0]))[0] == -5.0
    assert math.exp(oracle.log_decay(np.array([-200.0]))[0]) == 1.0   # alpha = 1 exactly
    # softplus(x) >= 5 exactly when x >= log(e^5 - 1) = 4.99321...
    thr = math.log(math.expm1(5.0))
    assert oracle.log_decay(np.array([thr + 1e-9]))[0] == -5.0
    assert oracle.log_decay(np.array([thr - 1e-6]))[0] > -5.0


def test_golden_paper_constants():
    c = _golden()
    keep, tol = c["floor_keep_fraction"]
    floor = oracle.log_decay(np.array([1e3]))[0]
    assert abs(math.exp(floor) - keep) <= tol             # 0.67% kept per step
    n = int(c["tile_tokens"][0])
    assert n == 16
    # all-floor tile: the cumulative log-decay reaches the low end exactly
    tile_sum = float(np.sum(oracle.log_decay(np.full(n, 1e3))))
    assert tile_sum == c["tile_logdecay_low"][0]
    # no decay at all: the high end
    assert float(np.sum(oracle.log_decay(np.full(n, -800.0)))) == c["tile_logdecay_high"][0]
    inv, tol = c["inverse_decay_bound"]
    assert abs(math.exp(-tile_sum) - inv) <= tol
    bmax, tol = c["bf16_max"]
    assert abs(float(torch.finfo(torch.bfloat16).max) - bmax) <= tol
    assert math.exp(-tile_sum) < float(torch.finfo(torch.bfloat16).max)
    # e^80 itself is representable in bf16 (finite after rounding)
    assert math.isfinite(float(torch.tensor(math.exp(80.0)).to(torch.bfloat16)))


# ---- P7: chunked form == token loop ----------------------------------------

@pytest.mark.parametrize("gmode", ["normal", "all_floor", "alpha_one", "mixed"])
@pytest.mark.parametrize("C", [1, 2, 4, 8, 16, 32, 64])
def test_p7_chunked_equals_recurrent(C, gmode):
    rng = np.random.default_rng(7 + C)
    T, dk, dv = 77, 16, 12
    q = rng.standard_normal((T, dk)); q /= np.linalg.norm(q, axis=1, keepdims=True)
    k = rng.standard_normal((T, dk)); k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, dv)); beta = rng.uniform(0, 1, T)
    s0 = rng.standard_normal((dk, dv)) * 0.5
    if gmode == "normal":
        g = rng.standard_normal((T, dk))
    elif gmode == "all_floor":
        g = np.full((T, dk), 30.0)
    elif gmode == "alpha_one":
        g = np.full((T, dk), -200.0)
    else:
        g = rng.standard_normal((T, dk)) * 8 + 2
    o_ref, S_ref = oracle.fwd_unit(q, k, v, g, beta, s0)
    o, S = chunk_mirror.forward_unit(q, k, v, g, beta, s0, chunk=C)
    assert np.max(np.abs(o - o_ref)) <= 1e-10 * max(1.0, np.max(np.abs(o_ref)))
    assert np.max(np.abs(S - S_ref)) <= 1e-10 * max(1.0, np.max(np.abs(S_ref)))


def test_p7_batched_varlen():
    rng = np.random.default_rng(70)
    lens = [1, 15, 16, 17, 63, 64, 65, 130]
    Tt, H, dk, dv = sum(lens), 2, 16, 8
    q = torch.from_numpy(rng.standard_normal((1, Tt, H, dk)))
    k = torch.nn.functional.normalize(torch.from_numpy(rng.standard_normal((1, Tt, H, dk))), dim=-1)
    v = torch.from_numpy(rng.standard_normal((1, Tt, H, dv)))
    g = torch.from_numpy(rng.standard_normal((1, Tt, H, dk)) * 3)
    beta = torch.from_numpy(rng.uniform(0, 1, (1, Tt, H)))
    s0 = torch.from_numpy(rng.standard_normal((len(lens), H, dk, dv)))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o1, S1 = oracle.fwd(q, k, v, g, beta, s0, cu_seqlens=cu)
    o2, S2 = chunk_mirror.forward(q, k, v, g, beta, s0, cu_seqlens=cu, chunk=64)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-10 * np.abs(o1).max())
    np.testing.assert_allclose(S2, S1, rtol=0, atol=1e-10 * np.abs(S1).max())
    # each packed sequence equals its own dense run
    for n, L in enumerate(lens):
        t0 = cu[n]
        od, Sd = oracle.fwd(q[:, t0:t0 + L], k[:, t0:t0 + L], v[:, t0:t0 + L],
                            g[:, t0:t0 + L], beta[:, t0:t0 + L], s0[n:n + 1])
        np.testing.assert_array_equal(od, o1[:, t0:t0 + L])
        np.testing.assert_array_equal(Sd, S1[n:n + 1])


def test_oracle_thread_count_invariant():
    rng = np.random.default_rng(5)
    B, T, H, dk, dv = 2, 40, 3, 8, 8
    args = [rng.standard_normal((B, T, H, dk)), rng.standard_normal((B, T, H, dk)),
            rng.standard_normal((B, T, H, dv)), rng.standard_normal((B, T, H, dk)),
            rng.uniform(0, 1, (B, T, H)), rng.standard_normal((B, H, dk, dv))]
    o1, S1 = oracle.fwd(*args, nthreads=1)
    o4, S4 = oracle.fwd(*args, nthreads=4)
    np.testing.assert_array_equal(o1, o4)
    np.testing.assert_array_equal(S1, S4)


# ---- P9: tile-bound invariant on the workloads' own inputs -----------------

@pytest.mark.parametrize("name", ["tiny_fp32", "h4_t4k", "b2_h32_t32k", "varlen_floor",
                                  "varlen_floor_hard"])
def test_p9_tile_bound_on_workloads(name):
    w = WORKLOADS[name]
    u = make_unit(w, 0, 0)
    g = u["g"].to(w.dtype)                      # the stored logits
    a = oracle.log_decay(g)
    assert a.min() >= -5.0 and a.max() <= 0.0
    T = a.shape[0]
    cuts = [0]
    if w.varlen:
        cuts = list(np.concatenate([[0], np.cumsum(w.seqlens())[:-1]]))
    worst = 0.0
    for s0, s1 in zip(cuts, cuts[1:] + [T]):
        for t0 in range(s0, s1, 16):
            tile = a[t0:min(t0 + 16, s1)].sum(axis=0)
            worst = min(worst, tile.min())
    assert -80.0 <= worst <= 0.0
    assert math.exp(-worst) <= math.exp(80.0) < float(torch.finfo(torch.bfloat16).max)
    frac = float((a == -5.0).mean())
    if name == "varlen_floor":
        # N(4,1) logits hit the floor only when x >= log(e^5-1) = 4.993: P ~ 0.160
        assert 0.15 < frac < 0.17, frac
    if name == "varlen_floor_hard":
        assert 0.83 < frac < 0.86, frac
        assert worst == -80.0


def test_varlen_lengths_recipe():
    w = WORKLOADS["varlen_floor"]
    lens = w.seqlens()
    assert sum(lens) == 32768
    assert all(128 <= L <= 4096 for L in lens)
    assert lens == w.seqlens()          # deterministic


# ---- the pins reject plausible mistakes ------------------------------------

def _mutant(kind):
    def f(q, k, v, g, beta, s0):
        q, k, v, g, beta = (np.asarray(t, dtype=np.float64) for t in (q, k, v, g, beta))
        T, dk = q.shape
        dv = v.shape[1]
        S = np.array(s0, dtype=np.float64)
        o = np.zeros((T, dv))
        for t in range(T):
            x = g[t]
            if kind == "no_floor":
                a = -np.logaddexp(0, x)
            elif kind == "softplus_sign":
                a = np.maximum(-np.logaddexp(0, -x), -5.0)
            elif kind == "floor_4":
                a = np.maximum(-np.logaddexp(0, x), -4.0)
            elif kind == "no_decay":
                a = np.zeros(dk)
            else:
                a = np.maximum(-np.logaddexp(0, x), -5.0)
            al = np.exp(a)
            if kind == "decay_after":
                p = S.T @ k[t]
                S = S + beta[t] * np.outer(k[t], v[t] - p)
                S = al[:, None] * S
            else:
                Sp = al[:, None] * S
                if kind == "read_before_decay":
                    p = S.T @ k[t]
                else:
                    p = Sp.T @ k[t]
                if kind == "beta_on_v_only":
                    S = Sp + np.outer(k[t], beta[t] * v[t] - p)
                elif kind == "drop_erase":
                    S = Sp + beta[t] * np.outer(k[t], v[t])
                else:
                    S = Sp + beta[t] * np.outer(k[t], v[t] - p)
            o[t] = S.T @ q[t]
        return o, S
    return f


def _mutant_prev_output():
    base = _mutant("none")

    def f(q, k, v, g, beta, s0):
        q = np.asarray(q, dtype=np.float64)
        T = q.shape[0]
        o = np.zeros((T, np.asarray(v).shape[1]))
        S = np.array(s0, dtype=np.float64)
        for t in range(T):
            o[t] = S.T @ q[t]                      # reads S_{t-1}
            _, S = base(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], beta[t:t + 1], S)
        return o, S
    return f


def _mutant_transposed_gate():
    base = _mutant("none")

    def f(q, k, v, g, beta, s0):
        # decay applied along the value axis instead of the key axis
        q, k, v, g, beta = (np.asarray(t, dtype=np.float64) for t in (q, k, v, g, beta))
        T, dk = q.shape
        dv = v.shape[1]
        S = np.array(s0, dtype=np.float64)
        o = np.zeros((T, dv))
        for t in range(T):
            al = np.exp(np.maximum(-np.logaddexp(0, g[t]), -5.0))
            Sp = S * al[None, :dv] if dv <= dk else S
            p = Sp.T @ k[t]
            S = Sp + beta[t] * np.outer(k[t], v[t] - p)
            o[t] = S.T @ q[t]
        return o, S
    return f


MUTANTS = {name: _mutant(name) for name in
           ["no_floor", "softplus_sign", "floor_4", "no_decay", "decay_after",
            "read_before_decay", "beta_on_v_only", "drop_erase"]}
MUTANTS["output_from_previous_state"] = _mutant_prev_output()
MUTANTS["decay_on_value_axis"] = _mutant_transposed_gate()


def test_reference_python_loop_passes_pins():
    f = _mutant("none")
    for pin in _pins.ALL:
        ok, err = pin(f)
        assert ok, (pin.__name__, err)


def _floor_pin(f):
    """All-floor gates: the state decays by exactly e^-5 per step (beta = 0)."""
    rng = np.random.default_rng(99)
    T, dk, dv = 6, 4, 3
    s0 = rng.standard_normal((dk, dv))
    q = rng.standard_normal((T, dk)); k = np.eye(dk)[[0, 1, 2, 3, 0, 1]]
    _, S = f(q, k, rng.standard_normal((T, dv)), np.full((T, dk), 40.0), np.zeros(T), s0)
    return np.allclose(S, np.exp(-5.0 * T) * s0, rtol=1e-12, atol=0)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name):
    f = MUTANTS[name]
    failed = [p.__name__ for p in _pins.ALL if not p(f)[0]]
    if not _floor_pin(f):
        failed.append("floor")
    assert failed, "mutant %s passed every pin" % name


def test_floor_pin_on_oracle():
    assert _floor_pin(c_unit)
    assert _floor_pin(mirror_unit(4))


# ---- the q scale -------------------------------------------------------------

def _c_scaled(q, k, v, g, beta, s0, scale):
    return oracle.fwd_unit(q, k, v, g, beta, s0, scale=scale)


def _mirror_scaled(C):
    def f(q, k, v, g, beta, s0, scale):
        return chunk_mirror.forward_unit(q, k, v, g, beta, s0, chunk=C, scale=scale)
    return f


def test_scale_pin_c_oracle():
    ok, err = _pins.p11_scale(_c_scaled)
    assert ok, err


@pytest.mark.parametrize("C", [1, 16, 64])
def test_scale_pin_chunk_mirror(C):
    ok, err = _pins.p11_scale(_mirror_scaled(C))
    assert ok, (C, err)


def test_scale_batched_oracle_is_linear_in_scale():
    # the batched entry (several heads, packed sequences) scales o only
    rng = np.random.default_rng(31)
    lens = [9, 40, 23]
    Tt, H, dk, dv = sum(lens), 2, 8, 4
    q = rng.standard_normal((1, Tt, H, dk)); k = rng.standard_normal((1, Tt, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, Tt, H, dv)); g = rng.standard_normal((1, Tt, H, dk))
    beta = rng.uniform(0, 1, (1, Tt, H)); s0 = rng.standard_normal((len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o1, S1 = oracle.fwd(q, k, v, g, beta, s0, cu_seqlens=cu)
    o2, S2 = oracle.fwd(q, k, v, g, beta, s0, cu_seqlens=cu, scale=-2.5)
    np.testing.assert_allclose(o2, -2.5 * o1, rtol=1e-14, atol=1e-14 * np.abs(o1).max())
    np.testing.assert_array_equal(S2, S1)
    o3, S3 = chunk_mirror.forward(q, k, v, g, beta, s0, cu_seqlens=cu, scale=-2.5)
    np.testing.assert_allclose(o3, o2, rtol=0, atol=1e-10 * np.abs(o2).max())
    np.testing.assert_allclose(S3, S2, rtol=0, atol=1e-10 * np.abs(S2).max())


def _scale_mutant(kind):
    base = _mutant("none")

    def f(q, k, v, g, beta, s0, scale):
        q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
        if kind == "scale_on_k":
            return base(q, k * scale, v, g, beta, s0)
        if kind == "scale_on_v":
            return base(q, k, v * scale, g, beta, s0)
        if kind == "scale_on_state":
            o, S = base(q, k, v, g, beta, s0)
            return o * scale, S * scale
        if kind == "scale_squared":
            return base(q * scale * scale, k, v, g, beta, s0)
        return base(q * scale, k, v, g, beta, s0)
    return f


def test_scale_pin_accepts_reference_loop():
    ok, err = _pins.p11_scale(_scale_mutant("none"))
    assert ok, err


@pytest.mark.parametrize("kind", ["scale_on_k", "scale_on_v", "scale_on_state",
                                  "scale_squared"])
def test_scale_pin_rejects_mutant(kind):
    ok, _ = _pins.p11_scale(_scale_mutant(kind))
    assert not ok, kind
