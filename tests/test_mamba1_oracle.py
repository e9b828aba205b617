"""Pins for the Mamba1 (per-channel state) part of the CPU oracle: an
independent matrix-form evaluation with a distinct decay rate per state
index, the reduction to the already pinned Mamba2 recurrence when a
channel's rates are all equal, hand-expanded arithmetic, closed forms for
A = 0 and Delta -> 0, and the chunk / decode invariants."""
import math

import numpy as np
import pytest

from tests import ssd_forms as F

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _case(rng, T, Dc, N, G, bias=(-4.0, -1.0)):
    x = rng.standard_normal((T, Dc))
    dt = rng.standard_normal((T, Dc))
    A = -np.exp(rng.uniform(-1.0, 2.0, (Dc, N)))
    B = rng.standard_normal((T, G, N))
    C = rng.standard_normal((T, G, N))
    D = rng.standard_normal(Dc)
    dt_bias = rng.uniform(bias[0], bias[1], Dc)
    return x, dt, A, B, C, D, dt_bias


@pytest.mark.parametrize("seed", [0, 1])
def test_mamba1_sequential_equals_matrix_form(oracle_lib, seed):
    """Every (channel, state index) pair has its own decay rate; the token
    recurrence equals the matrix form on two packed sequences with initial
    states, and the chunk-end states equal the matrix form's segment ends."""
    rng = np.random.default_rng(seed)
    lens, Dc, N, G = [37, 22], 6, 5, 2
    cu = np.array([0, 37, 59], np.int32)
    x, dt, A, B, C, D, dt_bias = _case(rng, 59, Dc, N, G)
    h0 = rng.standard_normal((2, Dc, N))
    cc = np.array([0, 16, 37, 50, 59], np.int32)
    y, cs, fs = oracle_lib.mamba1_prefill(x, dt, A, B, C, cu, cc, D=D, dt_bias=dt_bias, initial_states=h0)
    dl = F.deltas(dt, dt_bias)
    for r in range(2):
        a, b = cu[r], cu[r + 1]
        yq, endq = F.mamba1_quadratic(x[a:b], dl[a:b], A, B[a:b], C[a:b], D, h0[r])
        assert F.rel_err(y[a:b], yq) < 1e-12
        assert F.rel_err(fs[r], endq) < 1e-12
    _, mid = F.mamba1_quadratic(x[:16], dl[:16], A, B[:16], C[:16], D, h0[0])
    assert F.rel_err(cs[0], mid) < 1e-12
    assert F.rel_err(cs[1], fs[0]) < 1e-14 and F.rel_err(cs[3], fs[1]) < 1e-14


def test_mamba1_with_equal_rates_is_mamba2_with_headdim_one(oracle_lib):
    """With A[d, n] = a_d for every n, channel d is a Mamba2 head of headdim 1
    with scalar A_h = a_d: both oracle routines must agree (outputs, chunk
    states, final states)."""
    rng = np.random.default_rng(7)
    T, Dc, N, G = 45, 8, 4, 4
    cu = np.array([0, 20, 45], np.int32)
    cc = np.array([0, 7, 20, 31, 45], np.int32)
    x, dt, _, B, C, D, dt_bias = _case(rng, T, Dc, N, G)
    a = -np.exp(rng.uniform(0, 2, Dc))
    A = np.repeat(a[:, None], N, axis=1)
    h0 = rng.standard_normal((2, Dc, N))
    z = rng.standard_normal((T, Dc))
    y1, cs1, fs1 = oracle_lib.mamba1_prefill(x, dt, A, B, C, cu, cc, D=D, dt_bias=dt_bias, initial_states=h0, z=z)
    y2, cs2, fs2 = oracle_lib.ssd_prefill(x[:, :, None], dt, a, B, C, cu, cc, D=D, dt_bias=dt_bias,
                                          initial_states=h0[:, :, None, :], z=z[:, :, None])
    assert F.rel_err(y1, y2[:, :, 0]) < 1e-14
    assert F.rel_err(cs1, cs2[:, :, 0, :]) < 1e-14
    assert F.rel_err(fs1, fs2[:, :, 0, :]) < 1e-14


def test_mamba1_scalar_hand_expanded(oracle_lib):
    """Dc = N = G = 1: the scalar filter h_t = a_t h_{t-1} + b_t for three tokens."""
    A, Dd, bias = -0.7, -0.4, 0.1
    dts, xs, Bs, Cs, h0 = [0.5, -0.3, 1.2], [1.0, 2.5, -1.5], [0.6, -0.2, 1.4], [-1.0, 0.8, 0.3], -0.6
    d = [math.log(1.0 + math.exp(v + bias)) for v in dts]
    a = [math.exp(di * A) for di in d]
    b = [d[i] * xs[i] * Bs[i] for i in range(3)]
    h1 = a[0] * h0 + b[0]
    h2 = a[1] * h1 + b[1]
    h3 = a[2] * a[1] * a[0] * h0 + a[2] * a[1] * b[0] + a[2] * b[1] + b[2]
    yexp = [Cs[0] * h1 + Dd * xs[0], Cs[1] * h2 + Dd * xs[1], Cs[2] * h3 + Dd * xs[2]]
    y, _, fs = oracle_lib.mamba1_prefill(np.array(xs).reshape(3, 1), np.array(dts).reshape(3, 1),
                                         np.array([[A]]), np.array(Bs).reshape(3, 1, 1),
                                         np.array(Cs).reshape(3, 1, 1), [0, 3], D=np.array([Dd]),
                                         dt_bias=np.array([bias]), initial_states=np.array([[[h0]]]))
    assert np.allclose(y.ravel(), yexp, rtol=1e-14, atol=0)
    assert abs(fs.ravel()[0] - h3) < 1e-14


def test_mamba1_A_zero_is_prefix_sum(oracle_lib):
    """A = 0: no decay, so s_t[d,n] = h0[d,n] + sum_{s<=t} delta_s x_s[d] B_s[g,n]."""
    rng = np.random.default_rng(3)
    T, Dc, N, G = 30, 4, 3, 2
    x, dt, _, B, C, D, dt_bias = _case(rng, T, Dc, N, G)
    h0 = rng.standard_normal((1, Dc, N))
    y, _, fs = oracle_lib.mamba1_prefill(x, dt, np.zeros((Dc, N)), B, C, [0, T], D=D, dt_bias=dt_bias,
                                         initial_states=h0)
    dl = F.deltas(dt, dt_bias)
    grp = np.repeat(np.arange(G), Dc // G)
    Bd = B[:, grp, :]                                   # [T, Dc, N]
    s = h0[0][None] + np.cumsum((dl * x)[:, :, None] * Bd, axis=0)
    yexp = np.einsum("tdn,tdn->td", C[:, grp, :], s) + D[None, :] * x
    assert F.rel_err(y, yexp) < 1e-13
    assert F.rel_err(fs[0], s[-1]) < 1e-13


def test_mamba1_delta_to_zero_leaves_state(oracle_lib):
    """dt_bias = -100 makes Delta about 4e-44: the state stays h0 and y = C . h0 + D x."""
    rng = np.random.default_rng(4)
    T, Dc, N, G = 12, 4, 3, 1
    x, dt, A, B, C, D, _ = _case(rng, T, Dc, N, G)
    h0 = rng.standard_normal((1, Dc, N))
    y, _, fs = oracle_lib.mamba1_prefill(x, dt * 0.1, A, B, C, [0, T], D=D, dt_bias=np.full(Dc, -100.0),
                                         initial_states=h0)
    assert np.allclose(fs[0], h0[0], rtol=0, atol=1e-40)
    yexp = np.einsum("tn,dn->td", C[:, 0, :], h0[0]) + D[None, :] * x
    assert F.rel_err(y, yexp) < 1e-14


def test_mamba1_restart_from_chunk_state_equals_recompute(oracle_lib):
    """Prefix caching: the state stored at the end of chunk m, fed back as the
    initial state of the remaining tokens, reproduces the full run."""
    rng = np.random.default_rng(5)
    T, Dc, N, G, Q = 40, 4, 6, 2, 8
    x, dt, A, B, C, D, dt_bias = _case(rng, T, Dc, N, G)
    meta = oracle_lib.chunk_metadata([0, T], [0], Q)
    y, cs, fs = oracle_lib.mamba1_prefill(x, dt, A, B, C, [0, T], meta["cu_chunk_seqlens"], D=D, dt_bias=dt_bias)
    m = 3
    y2, _, fs2 = oracle_lib.mamba1_prefill(x[Q * m:], dt[Q * m:], A, B[Q * m:], C[Q * m:], [0, T - Q * m], D=D,
                                           dt_bias=dt_bias, initial_states=cs[m - 1][None])
    assert F.rel_err(y2, y[Q * m:]) < 1e-13
    assert F.rel_err(fs2, fs) < 1e-13


@pytest.mark.parametrize("null", [0, -1])
def test_mamba1_prefill_then_decode_equals_longer_prefill(oracle_lib, null):
    """Decoding two more tokens per request from the prefill's final state, through
    the cache routing (one padded row, spec columns), equals a longer prefill."""
    rng = np.random.default_rng(6)
    Dc, N, G, L, tpr = 4, 3, 1, 15, 2
    x, dt, A, B, C, D, dt_bias = _case(rng, L + tpr, Dc, N, G)
    y_full, _, fs_full = oracle_lib.mamba1_prefill(x, dt, A, B, C, [0, L + tpr], D=D, dt_bias=dt_bias)
    _, _, fs = oracle_lib.mamba1_prefill(x[:L], dt[:L], A, B[:L], C[:L], [0, L], D=D, dt_bias=dt_bias)
    cache = np.full((6, Dc, N), 7.0)
    cache[2] = fs[0]
    si = np.array([[2, 4], [null, null]], np.int32)
    xx = np.concatenate([x[L:], np.zeros((tpr, Dc))])
    dd = np.concatenate([dt[L:], np.zeros((tpr, Dc))])
    BB = np.concatenate([B[L:], np.zeros((tpr, G, N))])
    CC = np.concatenate([C[L:], np.zeros((tpr, G, N))])
    y, live, new = oracle_lib.mamba1_decode_with_cache(xx, dd, A, BB, CC, si, [0, 0], null, cache, D=D,
                                                       dt_bias=dt_bias)
    assert list(live) == [True, False]
    assert F.rel_err(y[:tpr], y_full[L:]) < 1e-13
    assert np.all(np.isnan(y[tpr:]))
    assert F.rel_err(new[4], fs_full[0]) < 1e-13
    keep = [i for i in range(6) if i not in (2, 4)]
    assert np.array_equal(new[keep], cache[keep])


@pytest.mark.parametrize("null", [0, -1])
def test_mamba1_cache_routing_hand_written(oracle_lib, null):
    """Slot routing of the Mamba1 state cache on hand-written slot lists
    ("[vLLM] Mamba (SSM) ...", "청크 메타데이터 계산": the state is taken out at
    every chunk end): sequence 0 resumes from slot 2, which its first chunk
    then overwrites (read before write); sequence 1 has a null initial slot
    (zero state); one chunk slot is null.  Expected values come from the
    independent matrix form, each segment started from the state the slot
    list names; slots no chunk writes keep their bits."""
    rng = np.random.default_rng(8)
    Dc, N, G = 4, 3, 1
    cu = [0, 13, 20]
    cc = [0, 5, 13, 16, 20]
    x, dt, A, B, C, D, dt_bias = _case(rng, 20, Dc, N, G)
    cache = rng.standard_normal((8, Dc, N))
    init_slot = [2, null]
    chunk_slot = [2, 5, null, 6]
    y, new = oracle_lib.mamba1_prefill_with_cache(x, dt, A, B, C, cu, cc, init_slot, chunk_slot, null,
                                                  cache, D=D, dt_bias=dt_bias)
    dl = F.deltas(dt, dt_bias)
    starts = [cache[2], np.zeros((Dc, N))]
    ends = []
    for r, segs in ((0, [(0, 5), (5, 13)]), (1, [(13, 16), (16, 20)])):
        h = starts[r]
        for a, b in segs:
            yq, h = F.mamba1_quadratic(x[a:b], dl[a:b], A, B[a:b], C[a:b], D, h)
            assert F.rel_err(y[a:b], yq) < 1e-12
            ends.append(h)
    assert F.rel_err(new[2], ends[0]) < 1e-12
    assert F.rel_err(new[5], ends[1]) < 1e-12
    assert F.rel_err(new[6], ends[3]) < 1e-12
    for s in (0, 1, 3, 4, 7):
        assert np.array_equal(new[s], cache[s]), s
